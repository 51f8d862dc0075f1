// Chunkwise prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// bf16 q/k/v, float32 state carried on chip from chunk to chunk.
//
// Two forms of the same arithmetic live here: the one-pass kernel described
// in this header (prefill_tc_kernel), and a two-pass form that the launcher
// takes when the workspace holds every chunk's key-side operands -- a
// key-side pass over all chunks of all sequences at once
// (prefill_prep_kernel), then the state recurrence loading those operands
// (prefill_state_kernel); both are described at their definitions below.
// The key-side steps are shared device functions, so the two forms give the
// same final states.
//
// One CTA owns one (b, h) sequence and walks its 64-token chunks.  With G_t
// the in-chunk cumulative log-decay, gamma_t = exp(G_t) and
// Gamma_ts = exp(G_t - G_s) (a difference, never a ratio of gammas):
//
//   A_ts = beta_t Gamma_ts (k_t . k_s) (s < t)     P_ts = Gamma_ts (q_t . k_s) (s <= t)
//   T    = (I + A)^{-1},  T' = T diag(beta gamma),  T'' = T diag(beta)
//   W^T  = K^T T'^T,      U~^T = V^T T''^T
//   U^T  = U~^T - S W^T          pseudo-values u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
//   O    = (diag(gamma) Q) S^T + P U
//   S   <- gamma_C S + U^T diag(exp(G_C - G_s)) K
//
// -- the token recurrence unrolled over a chunk (the pseudo-value rewriting
// of the delta rule, "On State Reduction in Linear Attention" notes, Sec. 2.3).
// Every product has M = 128 so that the accumulator row is the TMEM lane: the
// key-side and state products are written transposed (rows = value or key
// channels), and O is computed token-major from two stacked 64-row operands
// ([K; gamma Q] and [any 64 rows; P]) whose upper half is discarded, so each
// output row is one token's contiguous 256 bytes.
//
// Warp roles (16 warps, two warpgroups each):
//   key group   (warps 0-7): gates, A/P from [K;Q] K^T, the triangular
//               inverse T (16 x 16 blocks on CUDA cores), the W^T / U~^T
//               products and the -W^T operand; it also folds gamma into the Q
//               tile in place.  Thread 0 issues the V loads and these MMAs.
//               The key group depends on no state, so it runs up to one chunk
//               ahead of the state group.
//   state group (warps 8-15): U epilogue, state update, output.  Thread 256
//               issues the state-dependent MMAs and the q/k loads.
// The float32 state lives in state-group registers: thread (lane c, half h)
// holds row c, columns [h K/2, (h+1) K/2); a bf16 copy in shared memory is the
// MMA operand.  Register budgets are moved between the groups with
// setmaxnreg.  Groups hand off through mbarriers; every wait is bounded.
//
// Data movement: TMA loads 64-token x 64-channel bf16 boxes of q, k (three-stage
// ring) and v (single buffer) with the 128-byte swizzle; the same K tile is a
// K-major operand (contraction over channels) and an MN-major operand
// (contraction over tokens).  A ragged last chunk: TMA fills tokens past T
// with zeros; beta = 0 and log alpha = 0 there, which leaves valid rows
// unchanged.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"
#include "gdn_chunk.cuh"

#include <cudaTypedefs.h>

#include <algorithm>

namespace gdn {
namespace {

using namespace sm100;

constexpr int kKeyThreads = 256;
constexpr int kStateThreads = 256;
constexpr int kTcThreads = kKeyThreads + kStateThreads;
constexpr int kBarState = 2;  // named barrier id (kBarKey: the chunk helpers)

// Bytes of one chunk's key-side operands in the two-pass form: T'^T and
// T''^T, each a 64 x 64 bf16 tile stored as its 128-byte-swizzled
// shared-memory image.  (P, which needs q, is formed in the state pass from
// the q/k boxes it loads anyway.)
constexpr uint32_t kPrepTP = 0, kPrepTPP = 8192;
constexpr uint32_t kPrepChunkBytes = 16384;

// ---- the key-side steps of one chunk, shared by the fused kernel and the
// ---- separate key-side pass so that both compute bit-identical operands

// Gates of one chunk by one warp from alpha / beta held two per lane (tokens
// lane and lane + 32): G2 = in-chunk prefix of log2 alpha, gamma = 2^G2, beta.
__device__ __forceinline__ void chunk_gates(float pa0, float pa1, float pb0, float pb1, int lane,
                                            int nvalid, float *G2, float *gam, float *bet) {
    float g0, g1;
    chunk_log2_prefix(pa0, pa1, lane, nvalid, g0, g1);
    G2[lane] = g0;
    G2[lane + 32] = g1;
    gam[lane] = exp2f(g0);
    gam[lane + 32] = exp2f(g1);
    bet[lane] = pb0;
    bet[lane + 32] = pb1;
}

// [K;Q] K^T of one chunk into 64 TMEM columns at d1 (issued by one thread).
// The stage holds the 64-channel K and Q boxes adjacently (K at kc, Q at
// kc + 8 KB), so [K;Q] is one 128-row K-major operand.
template <int K>
__device__ __forceinline__ void issue_kq_kt(uint32_t d1, uint32_t stg, uint32_t kc0,
                                            uint32_t kc1) {
    constexpr uint32_t I_MM = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint32_t kb = ks / 4, ko = (ks % 4) * 32;
        const uint32_t kblk = stg + (kb ? kc1 : kc0) + ko;
        mma_bf16(d1, sdesc(kblk, 16, 1024), sdesc(kblk, 16, 1024), I_MM, ks > 0);
    }
}

// A_ts for s in [s0, s0 + 32) of row t (float32, into AF) from k_t . k_s in v
__device__ __forceinline__ void chunk_a_row(const float (&v)[32], int t, int s0,
                                            const float *G2, const float *bet, float *AF) {
    const float gt = G2[t], bt = bet[t];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 g = *reinterpret_cast<const float4 *>(G2 + s0 + i);
        const float gs[4] = {g.x, g.y, g.z, g.w};
        float a[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
            const int s = s0 + i + e2;
            a[e2] = s < t ? bt * decay_exp2(gt - gs[e2]) * v[i + e2] : 0.f;
        }
        *reinterpret_cast<float4 *>(AF + t * kLD + s0 + i) = make_float4(a[0], a[1], a[2], a[3]);
    }
}

// A (float32, rows 0..63 of AF) and P (bf16 operand tile) from [K;Q] K^T in
// TMEM; the thread holds TMEM lane quad_row, columns [32 colhalf, +32):
//   A_ts = beta_t 2^(G_t - G_s) (k_t . k_s) for s < t, else 0
//   P_ts = 2^(G_t - G_s) (q_t . k_s)       for s <= t, else 0
// Ptile may be shared or global memory (the tile's swizzled image), or null
// when no outputs are wanted.
__device__ __forceinline__ void chunk_ap(uint32_t taddr, int quad_row, int colhalf,
                                         const float *G2, const float *bet, float *AF,
                                         uint8_t *Ptile) {
    float v[32];
    tmem_ld32(taddr, v);
    tmem_ld_wait();
    const int t = quad_row & 63;
    const float gt = G2[t];
    const int s0 = 32 * colhalf;
    if (quad_row < 64) {
        chunk_a_row(v, t, s0, G2, bet, AF);
    } else if (Ptile != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const float4 g = *reinterpret_cast<const float4 *>(G2 + s0 + i);
            const float gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
                v[i + e2] = s0 + i + e2 <= t ? decay_exp2(gt - gs[e2]) * v[i + e2] : 0.f;
        }
        store_row<4>(Ptile, t, 4 * colhalf, v);
    }
}

// Block (i, j) of P from its product d (qk_block's layout) as bf16 pairs,
//   P_ts = 2^(G_t - G_s) (q_t . k_s) for s <= t, else 0
// (chunk_ap's P entries): w[nt][hr] holds t = 16 i + g + 8 hr and
// s = 16 j + 8 nt + 2 t4, +1 (g = lane / 4, t4 = lane % 4).
__device__ __forceinline__ void p_block_pack(const float (&d)[2][4], int i, int j, int lane,
                                             const float *G2, uint32_t (&w)[2][2]) {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int t = 16 * i + g + 8 * hr;
        const float gt = G2[t];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int s = 16 * j + 8 * nt + 2 * t4;
            const float2 gs = *reinterpret_cast<const float2 *>(G2 + s);
            const float x0 = s <= t ? decay_exp2(gt - gs.x) * d[nt][2 * hr] : 0.f;
            const float x1 = s + 1 <= t ? decay_exp2(gt - gs.y) * d[nt][2 * hr + 1] : 0.f;
            w[nt][hr] = pack_bf16(x0, x1);
        }
    }
}
// ... into the 128-byte-swizzled P tile (row t, s along the row)
__device__ __forceinline__ void p_block_store(uint8_t *tile, const uint32_t (&w)[2][2], int i,
                                              int j, int lane) {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
            *reinterpret_cast<uint32_t *>(tile + swz128(16 * i + g + 8 * hr, 2 * j + nt) +
                                          4 * t4) = w[nt][hr];
}
// The ten blocks of P on or below the diagonal, one per key-group warp (0-6)
// and a second for warps 0, 2 and 3 (warp 1 also forms the gates): block u
// is (i, j) = (3,0) (3,1) (3,2) (3,3) (2,0) (2,1) (2,2) (1,0) (1,1) (0,0).
__device__ __forceinline__ int p_unit_i(int u) { return u < 4 ? 3 : u < 7 ? 2 : u < 9 ? 1 : 0; }
__device__ __forceinline__ int p_unit_j(int u) { return u < 4 ? u : u < 7 ? u - 4 : u < 9 ? u - 7 : 0; }
__device__ __forceinline__ int p_extra_unit(int warp) {
    return warp == 0 ? 7 : warp == 2 ? 8 : warp == 3 ? 9 : -1;
}

// Which token range, initial state and final-state slot a CTA works on.
//   kWhole:  CTA = one (b, h) sequence, tokens [0, T), S0 / S_T as given.
//   kFirst:  long sequences cut into `nseg` segments of `seg_len` tokens; per
//            sequence 2 nseg - 1 CTAs: segment 0 from S0 with outputs (its end
//            state into slot E), and for each later segment p the end state
//            from a zero start (slot H) and the transition matrix (slot M: the
//            same recurrence run on the rows of the identity with v = 0).
//   kSecond: segments p >= 1 again from their start states (slot S, filled by
//            the combine kernel) with outputs; the last one writes S_T.
//   kFirstX: kFirst with every run writing outputs: the zero-start runs o0 of
//            their segment into o, the identity-start runs (v = 0) X into the
//            X buffer; o = o0 + S_start X^T then replaces the second pass.
// The end state of a segment is affine in its start state (the update is
// S -> alpha S (I - beta k k^T) + beta v k^T), so S_end = S_start M + H; so
// is every output of the segment: o_t = o0_t + S_start x_t, where x_t is the
// output of the same recurrence run on the rows of the identity with v = 0.
enum SegMode : int { kWhole = 0, kFirst = 1, kSecond = 2, kFirstX = 3 };
struct SegPlan {
    int mode;
    int nseg;
    int seg_len;  // multiple of 64
    float *ws;    // [3][B*H][nseg][V][K]: H/E slots, M slots, start-state slots
};

struct SegTask {
    size_t seq;        // (b, h) sequence
    int t0, t1;        // token range
    const float *s0p;  // start state (nullptr: zero)
    bool s0_identity;  // start from the identity (transition-matrix run)
    float *stp;        // end-state destination (nullptr: none)
    bool zero_v;       // v = 0 (transition-matrix run)
    bool outputs;      // this run writes o
    bool out_x;        // ... into the X buffer instead
};
__device__ __forceinline__ SegTask segment_task(const SegPlan &plan, int K, int T,
                                                const float *S0, float *ST, int BH) {
    constexpr int V = 128;
    const size_t VK = (size_t)V * K;
    SegTask tk{blockIdx.x, 0, T, nullptr, false, nullptr, false, true, false};
    if (plan.mode == kWhole) {
        if (S0) tk.s0p = S0 + tk.seq * VK;
        if (ST) tk.stp = ST + tk.seq * VK;
        return tk;
    }
    auto slot = [&](int kind, size_t sq, int p) {
        return plan.ws + ((kind * (size_t)BH + sq) * plan.nseg + p) * VK;
    };
    int p;
    if (plan.mode == kFirst || plan.mode == kFirstX) {
        const bool x = plan.mode == kFirstX;
        tk.seq = blockIdx.x / (2 * plan.nseg - 1);
        const int i = blockIdx.x % (2 * plan.nseg - 1);
        p = (i + 1) / 2;
        if (i == 0) {
            if (S0) tk.s0p = S0 + tk.seq * VK;
            tk.stp = slot(0, tk.seq, 0);  // end of segment 0 (E)
        } else if (i & 1) {
            tk.stp = slot(0, tk.seq, p);  // zero start: H (and o0)
            tk.outputs = x;
        } else {
            tk.s0_identity = true;        // identity start, v = 0: M (and X)
            tk.zero_v = true;
            tk.stp = slot(1, tk.seq, p);
            tk.outputs = x;
            tk.out_x = x;
        }
    } else {
        tk.seq = blockIdx.x / (plan.nseg - 1);
        p = 1 + blockIdx.x % (plan.nseg - 1);
        tk.s0p = slot(2, tk.seq, p);
        tk.stp = (p == plan.nseg - 1 && ST) ? ST + tk.seq * VK : nullptr;
    }
    tk.t0 = p * plan.seg_len;
    tk.t1 = min(T, tk.t0 + plan.seg_len);
    return tk;
}

// ---------------------------------------------------------------- key-side pass
// The two-pass form's first kernel.  Everything of a chunk that depends only
// on its keys and gates -- A, the inverse T and T', T'' -- has no dependence
// on the state, so it runs for all B * H * ceil(T/64) chunks at once instead
// of in each sequence's serial chunk loop.  Persistent CTAs of 128 threads
// (four per SM, so that one CTA's loads and waits hide under the others'
// work) stride over the chunks; each chunk's K K^T is one tcgen05 product
// into 64 TMEM columns (the [K;Q] operand of the fused kernel with a zero Q
// half: q is not read here), the next chunk's k boxes load (TMA) while the
// current one is solved, and T'^T and T''^T go to global memory as their
// swizzled shared-memory images, which the state-side kernel copies in with
// bulk copies.  Same arithmetic as the fused kernel's key group (the shared
// helpers above), so both forms give identical states.  The gathering form
// loads the full-width q and k boxes, and writes the gathered q' and k' for
// the state pass.
// The product reads 128 rows of its A operand, [K;Q] in the fused kernel's
// layout; here only the K rows (TMEM lanes 0..63) are used, so lanes 64..127
// may hold anything, and rows 64..127 of A are whatever lies 8 KB past each
// box: the next k box, or the start of the A scratch (written only between
// the products, after the previous one has completed).  The stage then holds
// just the k boxes.  The gathering form loads the full-width q and k boxes.
template <int K, bool GATHER>
struct PrepLayout {
    // gathering: the q and k boxes of all 128 channels.  Otherwise each k box
    // is loaded twice, 8 KB apart, so that the product's A operand (128 rows)
    // is [K; K] and TMEM lanes 64..127 hold K K^T again
    static constexpr uint32_t KC0 = 0, QC0 = 8192, KDUP = 8192;
    static constexpr uint32_t KC1 = 16384, QC1 = 24576;  // KC1: K = 128 or gathering
    static constexpr uint32_t STAGE = (GATHER || K == 128) ? 32768 : 16384;
    static constexpr uint32_t AF = STAGE;                  // float [64][68]
    static constexpr uint32_t GATE = AF + 64 * kLD * 4;    // G2, gamma, beta
    static constexpr uint32_t END = GATE + 3 * 64 * 4;
    static constexpr uint32_t KQ_BYTES = 4u * 8192u;
    static constexpr uint32_t K_BYTES = (K == 128 ? 4u : 2u) * 8192u;
    static constexpr size_t SMEM = END;
    static_assert(GATHER || STAGE >= (K == 128 ? KC1 : KC0) + 16384, "[K; K] of the last box");
    static_assert(!GATHER || 64 * kLD * 4 >= 16384, "the A scratch holds the gathered [K'; K']");
};
constexpr int kPrepThreads = 128;
// resident CTAs per SM (five or six with the k-only stage ran slower: the
// register budget they leave spills the inverse)
constexpr int prep_ctas_per_sm(bool) { return 4; }
// the CTAs' dynamic + 1 KB static + 1 KB reserved shared memory per SM
static_assert(prep_ctas_per_sm(false) * (PrepLayout<128, false>::SMEM + 2048) <= 233472,
              "prep residency");
static_assert(prep_ctas_per_sm(true) * (PrepLayout<64, true>::SMEM + 2048) <= 233472,
              "prep residency");

// The pruning prologue inside the key-side pass (GATHER): the q/k boxes are
// the full 128-channel rows, the kernel keeps channels idx[h, :] of each row
// and renormalises them over the kept channels, feeds the gathered [K';Q'] to
// its own products and writes q', k' ([B, T, H, 64] bf16) for the state pass.
struct PrepGather {
    const int *idx;      // [H, 64] kept channels of each head
    __nv_bfloat16 *qg;   // [B, T, H, 64] gathered, renormalised q
    __nv_bfloat16 *kg;   // [B, T, H, 64] gathered, renormalised k
};

template <int K, bool GATHER>
__global__ void __launch_bounds__(kPrepThreads, prep_ctas_per_sm(GATHER))
    prefill_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const float *__restrict__ alpha,
                        const float *__restrict__ beta, uint8_t *__restrict__ prep, int T, int Ts,
                        int H, long long nchunk_all, PrepGather gth, int *status) {
    static_assert(!GATHER || K == 64, "the gathering form keeps 64 of 128 channels");
    using L = PrepLayout<K, GATHER>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzle atoms and operand descriptors need a 1024-byte aligned
    // base; the declaration provides it and the kernel checks it
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && status) atomicOr(status, kStatusBounds);
        return;
    }
    uint8_t *sm = smem_raw;
    __shared__ uint64_t kq_full, bar_p1, drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int *abort_v = &abort_flag;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nch = (T + 63) / 64;  // chunks per sequence

    // the state pass may be scheduled now (it waits for this grid before
    // reading the operands; every CTA of this persistent grid is resident)
    if (tid == 0) pdl_trigger();
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_init(&kq_full, 1);
        mbar_init(&bar_p1, 1);
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int quad_row = (warp & 3) * 32 + lane;
    float *AF = reinterpret_cast<float *>(sm + L::AF);
    float *G2 = reinterpret_cast<float *>(sm + L::GATE);
    float *gam = G2 + 64;
    float *bet = G2 + 128;

    // item j of the persistent loop: chunk n of sequence seq, taken in
    // reverse chunk-major order (chunk nch - 1 of every sequence first), so
    // that the operands the state pass reads first are the ones written last,
    // still in L2 when it starts
    const long long BHs = nchunk_all / nch;
    auto item = [&](long long j, long long &seq, int &n) {
        seq = j % BHs;
        n = nch - 1 - (int)(j / BHs);
    };
    auto load_kq = [&](long long j) {
        if (!bounds_ok(j >= 0 && j < nchunk_all, status)) return;
        long long seq;
        int n;
        item(j, seq, n);
        const int b = (int)(seq / H), h = (int)(seq % H);
        // the gathering form loads q and k, both with all 128 channels
        mbar_arrive_expect_tx(&kq_full, GATHER ? L::KQ_BYTES : L::K_BYTES);
        tma_load_4d(sm + L::KC0, &tm_k, &kq_full, 0, h, n * 64, b);
        if (GATHER) tma_load_4d(sm + L::QC0, &tm_q, &kq_full, 0, h, n * 64, b);
        else tma_load_4d(sm + L::KC0 + L::KDUP, &tm_k, &kq_full, 0, h, n * 64, b);
        if (K == 128 || GATHER) {
            tma_load_4d(sm + L::KC1, &tm_k, &kq_full, 64, h, n * 64, b);
            if (GATHER) tma_load_4d(sm + L::QC1, &tm_q, &kq_full, 64, h, n * 64, b);
            else tma_load_4d(sm + L::KC1 + L::KDUP, &tm_k, &kq_full, 64, h, n * 64, b);
        }
    };
    float pa0 = 1.f, pa1 = 1.f, pb0 = 0.f, pb1 = 0.f;  // prefetched gate inputs (warp 1)
    auto prefetch_gates = [&](long long j) {
        if (warp == 1 && j < nchunk_all && bounds_ok(T <= Ts, status)) {
            long long seq;
            int n;
            item(j, seq, n);
            const int b = (int)(seq / H), h = (int)(seq % H);
            const int nv = min(64, T - n * 64);
            const size_t i0 = ((size_t)b * Ts + n * 64 + lane) * H + h;
            const size_t i1 = i0 + (size_t)32 * H;
            pa0 = lane < nv ? alpha[i0] : 1.f;
            pb0 = lane < nv ? beta[i0] : 0.f;
            pa1 = lane + 32 < nv ? alpha[i1] : 1.f;
            pb1 = lane + 32 < nv ? beta[i1] : 0.f;
        }
    };
    // bounded wait that sleeps between polls: other CTAs on the SM are busy
    // with shared memory, which a tight poll would take cycles from
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

    const long long G = gridDim.x;
    long long j = blockIdx.x;
    if (tid == 0 && j < nchunk_all) load_kq(j);
    prefetch_gates(j);
    bool failed = false;
    for (int it = 0; j < nchunk_all; j += G, ++it) {
        long long seq;
        int n;
        item(j, seq, n);
        const int nvalid = min(64, T - n * 64);
        bool ok = true;
        if constexpr (GATHER) {
            if (tid == 0) ok = wait(&kq_full, it & 1);
            if (named_sync_or(kBarKey, kPrepThreads, !ok)) { failed = true; break; }
            // eight lanes per row, eight kept channels per lane (channels
            // 8 cl .. 8 cl + 7 of idx[h]), four rows per warp pass: warp w owns
            // rows 32 w .. 32 w + 31 of [K'; Q'] (K tokens, then Q tokens).  The
            // sum of squares runs in the standalone prologue's order (eight
            // channels per lane, then the lanes 4, 2, 1 apart), so the rows are
            // bit-identical to gdn_gather_normalize
            const int h = (int)(seq % H), b = (int)(seq / H);
            const int sub = lane >> 3, cl = lane & 7;
            const int4 *ip = reinterpret_cast<const int4 *>(gth.idx + (size_t)h * 64) + 2 * cl;
            const int4 i0 = __ldg(ip), i1 = __ldg(ip + 1);
            const int cs[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
            bool bad = false;
            uint8_t *tile = sm + L::AF;  // [K';K'] in the A scratch, read before A is written
#pragma unroll 1
            for (int pass = 0; pass < 8; ++pass) {
                const int r = 32 * warp + 4 * pass + sub;  // row of [K'; Q']
                const int t = r & 63;
                const uint8_t *src = sm + (r < 64 ? L::KC0 : L::QC0);  // channels 64..127: +16 KB
                float gv[8], ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = cs[e];
                    float x = 0.f;
                    if ((unsigned)c < 128u) {
                        const int cc = c & 63;
                        x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                            src + (c >> 6) * 16384 + swz128(t, cc >> 3) + (cc & 7) * 2));
                    } else {
                        bad = true;
                    }
                    gv[e] = x;
                    ss = fmaf(x, x, ss);
                }
#pragma unroll
                for (int off = 4; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
                uint4 w;
                w.x = pack_bf16(gv[0] * inv, gv[1] * inv);
                w.y = pack_bf16(gv[2] * inv, gv[3] * inv);
                w.z = pack_bf16(gv[4] * inv, gv[5] * inv);
                w.w = pack_bf16(gv[6] * inv, gv[7] * inv);
                // the tile is [K'; K'] (A's 128 rows), the q' rows go out only
                if (r < 64) {
                    *reinterpret_cast<uint4 *>(tile + swz128(r, cl)) = w;
                    *reinterpret_cast<uint4 *>(tile + swz128(r + 64, cl)) = w;
                }
                if (t < nvalid && bounds_ok(seq < nchunk_all / nch && n * 64 + t < T, status))
                    reinterpret_cast<uint4 *>((r < 64 ? gth.kg : gth.qg) +
                                              (((size_t)b * T + (size_t)n * 64 + t) * H + h) * 64)[cl] =
                        w;
            }
            if (bad && status) atomicOr(status, kStatusBounds);
            // the tile feeds the product; the stage's reads precede its reload
            fence_proxy_async_smem();
            named_sync(kBarKey, kPrepThreads);
            if (tid == 0) {
                if (j + G < nchunk_all) load_kq(j + G);
                tc_fence_after();
                issue_kq_kt<K>(tb, smem_u32(sm) + L::AF, 0, 0);
                mma_commit(&bar_p1);
                ok = wait(&bar_p1, it & 1);
            }
        } else {
            if (tid == 0) {
                ok = wait(&kq_full, it & 1);
                if (ok) {
                    tc_fence_after();
                    issue_kq_kt<K>(tb, smem_u32(sm), L::KC0, L::KC1);
                    mma_commit(&bar_p1);
                    ok = wait(&bar_p1, it & 1);
                    // the product has read the stage: the next chunk's boxes may land
                    if (ok && j + G < nchunk_all) load_kq(j + G);
                }
            }
        }
        if (warp == 1) {
            chunk_gates(pa0, pa1, pb0, pb1, lane, nvalid, G2, gam, bet);
            prefetch_gates(j + G);
        }
        if (named_sync_or(kBarKey, kPrepThreads, !ok)) { failed = true; break; }
        uint8_t *out = prep + ((size_t)seq * nch + n) * kPrepChunkBytes;  // [T'^T | T''^T]
        tc_fence_after();
        {   // lanes 64..127 repeat K K^T: warps 0-1 form columns 0..31 of A's
            // rows, warps 2-3 columns 32..63
            const int ch = warp >> 1, t = quad_row & 63;
            float v[32];
            tmem_ld32(tb + lane_off + 32 * ch, v);
            tmem_ld_wait();
            chunk_a_row(v, t, 32 * ch, G2, bet, AF);
        }
        tc_fence_before();
        named_sync(kBarKey, kPrepThreads);
        chunk_inverse_tprime<kPrepThreads>(AF, bet, gam, out + kPrepTP, out + kPrepTPP, tid);
        named_sync(kBarKey, kPrepThreads);  // AF and the gates are rewritten next
    }

    if (failed) *abort_v = 1;
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        if (tid == 0) {
            if (status) atomicOr(status, kStatusTimeout);
            // a product still in flight reads shared memory and writes TMEM
            mma_commit(&drain);
            mbar_wait(&drain, 0, kSpinLimit / 16);
            // let an in-flight load land before the CTA's shared memory is released
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

// ---------------------------------------------------------------- state-side pass
// The two-pass form's second kernel: one CTA per (b, h) sequence (or segment)
// walks its chunks like the fused kernel, but loads T'^T and T''^T instead
// of solving for them.  Three roles:
//   key group (warps 0-6): per chunk P = (Q K^T masked, times the decays)
//       with warp-level MMAs from the raw q/k boxes (forming P here saves the
//       key-side pass its q read and P's trip through memory), the gates,
//       the state group's decay factors and gamma folded into the Q box (no
//       tensor-memory products, no loads).  It runs up to a chunk ahead of
//       the state group.
//   issuer (warp 7, one thread): every TMA load, and the products off the
//       state chain -- O^T(n) = S(n-1) (gamma Q(n))^T once the state thread
//       has issued U(n) (it runs behind it), then, once U(n) is complete,
//       W^T(n+1) = K^T T'^T and U~^T(n+1) = V^T T''^T (its U slot was
//       U(n-1)'s) -- while the chain's epilogue leaves the tensor pipe idle.
//       An SM issues tcgen05 products one at a time, so the chain's own
//       products are never issued beside these.
//   state group (warps 8-15): the state chain
//       U^T(n)  = U~^T(n) + S(n-1) (-W^T(n))       (issued at the end of n - 1)
//       epilogue: U^T -> bf16, U^T diag(decay) -> bf16, in the U slot
//       dS(n)   = U^T diag(decay) K(n),  O^T(n) += U^T P(n)^T
//       -W^T(n+1) from TMEM into its operand tile, while dS(n) runs
//       S(n)    = gamma_C S(n-1) + dS(n)
//     and the transposed output, staged by warps 12-15 for TMA stores by
//     warp 11 (a ragged tail is clipped by the tensor map).
// The chain's A operands live in TMEM (the bf16 state, and bf16 U^T and
// U^T diag(decay) written back into the spent U accumulator), so its products
// read only their B operands from shared memory.  Ordering: a commit covers
// every earlier product of its thread, so bar_u(n) (the state thread's
// commit after U(n)) also says that dS(n-1) and O^T(n-1) += U^T P^T are
// complete: the issuer reloads and reuses slots only after it.  The state
// thread waits for the S-term (bar_os), which reads S(n-1), before its
// O^T(n) += U^T P^T and the update, for U~^T(n) (bar_ut) before U(n), and
// for the key group's chunk n (key_ready(n): decays, P(n), gamma Q(n)) before
// the epilogue of chunk n; the issuer writes W^T(n+1) only after the state
// group has read W^T(n) (u_sig(n) follows it).  The key group stores P(n)
// once O^T(n-1) += U^T P^T is complete (bar_o2), and with it O^T(n-2)'s,
// the last reader of the slot.
// Every mbarrier wait is for the barrier's latest phase: the next phase needs
// a step that the waiting thread takes after the wait (key_ready is a ring of
// four because the key group may run ahead).  Rings: q/k (three stages), V,
// [T'^T | T''^T], P, U and O (two each); the loads of chunk n + 2 go out in
// chunk n's window.  Every state quantity is the fused kernel's arithmetic on
// the same operands, so S_T is bit-identical to it (o agrees to the
// accumulation orders of P and of the transposed product).

// Rings: K and Q (three slots each), V, [T'^T | T''^T] and P (two each);
// one -W^T tile.  Each K / Q slot holds the 64-channel boxes of one chunk
// side by side (channels 64..127 at +8 KB when K = 128).
template <int K>
struct StLayout {
    static constexpr int NK = 3, NQ = 3, NV = 2, NT = 2;
    static constexpr uint32_t BOX = K == 128 ? 16384 : 8192;     // one chunk of k or q
    static constexpr uint32_t KR = 0;                            // K ring
    static constexpr uint32_t QR = KR + NK * BOX;                // Q ring
    static constexpr uint32_t VB = QR + NQ * BOX;                // V ring, 16 KB per chunk
    static constexpr uint32_t PR = VB + NV * 16384;              // ring of [T'^T | T''^T]
    static constexpr uint32_t PP = PR + NT * 16384;              // ring of P
    static constexpr uint32_t OST = PP + 2 * 8192;               // output staging, 2 x 64 x 64
    static constexpr uint32_t NWB = OST + 16384;                 // -W^T, K x 64
    static constexpr uint32_t KGATE = NWB + 16384;               // G2, gamma, beta
    static constexpr uint32_t SGATE = KGATE + 3 * 64 * 4;        // 3 x (decay[64], gamma_C)
    static constexpr uint32_t END = SGATE + 3 * 68 * 4;
    static constexpr uint32_t V_BYTES = 2u * 8192u;
    static constexpr size_t SMEM = END;
    static_assert(SMEM + 1024 <= 232448, "shared memory budget");
    static __device__ __forceinline__ uint32_t kbuf(int n) { return KR + (n % NK) * BOX; }
    static __device__ __forceinline__ uint32_t qbuf(int n) { return QR + (n % NQ) * BOX; }
    static __device__ __forceinline__ uint32_t tp(int n) { return PR + (n % NT) * 16384; }
    static __device__ __forceinline__ uint32_t tpp(int n) { return tp(n) + 8192; }
    static __device__ __forceinline__ uint32_t ptile(int n) { return PP + (n & 1) * 8192; }
    static __device__ __forceinline__ uint32_t vbuf(int n) { return VB + (n % NV) * 16384; }
    // TMEM columns: O^T of even / odd chunks, U~^T / U^T of even / odd
    // chunks, the bf16 state (two K elements per column), W^T, dS
    static constexpr uint32_t O0 = 0, O1 = 64, UA = 128, SBT = 256, WT = 320, DS = 384;
    static __device__ __forceinline__ uint32_t ocol(int n) { return (n & 1) ? O1 : O0; }
    static __device__ __forceinline__ uint32_t ua(int n) { return UA + 64 * (n & 1); }
    // After chunk n's epilogue, token half h of its U slot (32 columns) holds
    // bf16 U^T in its first 16 columns and bf16 U^T diag(decay) in the next
    // 16: the TMEM A operand of K step ks (16 tokens) of O^T += U^T P^T / dS.
    static __device__ __forceinline__ uint32_t ut_col(int n, int ks) {
        return ua(n) + 32 * (ks >> 1) + 8 * (ks & 1);
    }
    static __device__ __forceinline__ uint32_t ud_col(int n, int ks) { return ut_col(n, ks) + 16; }
};

constexpr int kBarOut = 3, kBarOut2 = 4;  // the output warps (11-15)
constexpr int kStKeyThreads = 224;        // warps 0-6
constexpr int kStIssuer = 224;            // warp 7, lane 0

template <int K>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_state_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o,
                         const __grid_constant__ CUtensorMap tm_x, const float *__restrict__ alpha,
                         const float *__restrict__ beta, const float *__restrict__ S0,
                         bool want_o, float *__restrict__ ST, int T, int Ts, int H, int BH,
                         SegPlan plan, const uint8_t *__restrict__ prep, int *status) {
    using L = StLayout<K>;
    constexpr int KH = K / 2;  // state columns per state-group thread
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && status) atomicOr(status, kStatusBounds);
        return;
    }
    uint8_t *sm = smem_raw;
    __shared__ uint64_t k_full[3], q_full[3], v_full[2], tt_full[2], key_ready[4], bar_w, bar_ut,
        bar_u, bar_s, bar_os, bar_o2, u_sig, drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int *abort_v = &abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const SegTask tk = segment_task(plan, K, T, S0, ST, BH);
    // (every thread takes the same branch, before any barrier or allocation)
    if (!bounds_ok(tk.seq < (size_t)BH && tk.t0 >= 0 && tk.t0 < tk.t1 && tk.t1 <= T &&
                       tk.t0 % 64 == 0 && T <= Ts,
                   status))
        return;
    const size_t seq = tk.seq;
    const int t0 = tk.t0, t1 = tk.t1;
    const bool zero_v = tk.zero_v;
    const bool outs = want_o && tk.outputs;
    const CUtensorMap *tm_out = tk.out_x ? &tm_x : &tm_o;  // where the outputs go
    const int b = (int)(seq / H), h = (int)(seq % H);
    const int nchunks = (t1 - t0 + 63) / 64;
    const uint32_t base = smem_u32(sm);
    // -W^T, T''^T, P of chunk n of this CTA's token range
    const uint8_t *prep_seq = prep + (seq * (size_t)((T + 63) / 64) + t0 / 64) * kPrepChunkBytes;

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        uint64_t *bars[] = {&k_full[0],  &k_full[1],  &k_full[2],  &q_full[0],  &q_full[1],
                            &q_full[2],  &v_full[0],  &v_full[1],  &tt_full[0], &tt_full[1],
                            &key_ready[0], &key_ready[1], &key_ready[2], &key_ready[3],
                            &bar_w,    &bar_ut,     &bar_u,  &bar_s,  &bar_os,
                            &u_sig,      &bar_o2,     &drain[0],   &drain[1]};
        for (uint64_t *bb : bars) mbar_init(bb, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int quad_row = (warp & 3) * 32 + lane;  // TMEM lane of this thread
    // decay[64] and gamma_C of chunk n in slot n % 3 (written by the key group)
    float *sg = reinterpret_cast<float *>(sm + L::SGATE);

    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_or_abort(bar, parity, kSpinLimit, abort_v);
        if (!ok) *abort_v = 1;
        return ok;
    };

    constexpr uint32_t I_MM = idesc_bf16(128, 64, false, false);  // K-major x K-major, N = 64
    constexpr uint32_t I_ABMN = idesc_bf16(128, 64, true, true);  // MN-major A and B
    constexpr uint32_t I_BMN = idesc_bf16(128, 64, false, true);  // MN-major B, N = 64
    constexpr uint32_t I_DS = idesc_bf16(128, K, false, true);    // MN-major B, N = K

    bool failed = false;

    if (tid < kStKeyThreads) {
        // ================================================================ key group
        asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
        float *G2 = reinterpret_cast<float *>(sm + L::KGATE);
        float *gam = G2 + 64;
        float *bet = G2 + 128;
        // gate inputs of chunks n and n + 1 in warp 1's registers: each
        // chunk's alpha / beta are loaded two iterations before they are
        // used, so the load latency stays off the key group's loop
        float pa[2][2] = {{1.f, 1.f}, {1.f, 1.f}}, pb[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        auto prefetch_gates = [&](int n, int slot) {
            if (warp == 1 && n < nchunks) {
                const int nv = min(64, t1 - t0 - n * 64);
                const size_t i0 = ((size_t)b * Ts + t0 + n * 64 + lane) * H + h;
                const size_t i1 = i0 + (size_t)32 * H;
                pa[slot][0] = lane < nv ? alpha[i0] : 1.f;
                pb[slot][0] = lane < nv ? beta[i0] : 0.f;
                pa[slot][1] = lane + 32 < nv ? alpha[i1] : 1.f;
                pb[slot][1] = lane + 32 < nv ? beta[i1] : 0.f;
            }
        };
        prefetch_gates(0, 0);
        prefetch_gates(1, 1);
        // P's blocks above the diagonal stay zero in both ring slots
        if (outs)
            for (int e = tid; e < 2 * 8192 / 16; e += kStKeyThreads)
                reinterpret_cast<uint4 *>(sm + L::PP)[e] = make_uint4(0u, 0u, 0u, 0u);
        const int pu2 = p_extra_unit(warp);
        for (int n = 0; n < nchunks; ++n) {
            const int p2 = n & 1;
            const int nvalid = min(64, t1 - t0 - n * 64);
            bool ok = true;
            if (tid == 0)
                ok = wait(&q_full[n % L::NQ], (n / L::NQ) & 1) &&
                     wait(&k_full[n % L::NK], (n / L::NK) & 1);
            if (named_sync_or(kBarKey, kStKeyThreads, !ok)) { failed = true; break; }
            // P(n) = (Q K^T) from the raw boxes, before Q is scaled in place
            float pd[2][2][4];
            if (outs) {
                const uint32_t qb = base + L::qbuf(n), kb = base + L::kbuf(n);
                qk_block<K>(qb, qb + 8192, kb, kb + 8192, p_unit_i(warp), p_unit_j(warp), lane,
                            pd[0]);
                if (pu2 >= 0)
                    qk_block<K>(qb, qb + 8192, kb, kb + 8192, p_unit_i(pu2), p_unit_j(pu2), lane,
                                pd[1]);
            }
            if (warp == 1) {
                if (p2 == 0)
                    chunk_gates(pa[0][0], pa[0][1], pb[0][0], pb[0][1], lane, nvalid, G2, gam, bet);
                else
                    chunk_gates(pa[1][0], pa[1][1], pb[1][0], pb[1][1], lane, nvalid, G2, gam, bet);
                __syncwarp();
                // the state group's decay to the chunk end and gamma_C; slot
                // n % 3 was last read in the state epilogue of chunk n - 3,
                // which precedes U(n - 2) and so the load of this chunk's q box
                float *slot = sg + (n % 3) * 68;
                const float gC = G2[63];
                slot[lane] = exp2f(gC - G2[lane]);
                slot[lane + 32] = exp2f(gC - G2[lane + 32]);
                if (lane == 0) slot[64] = exp2f(gC);
            }
            named_sync(kBarKey, kStKeyThreads);  // gates in place; raw Q read
            uint32_t pw[2][2][2];
            if (outs) {
                p_block_pack(pd[0], p_unit_i(warp), p_unit_j(warp), lane, G2, pw[0]);
                if (pu2 >= 0) p_block_pack(pd[1], p_unit_i(pu2), p_unit_j(pu2), lane, G2, pw[1]);
            }
            // Q <- diag(gamma) Q in place (next read by the O^T S-term)
            for (int e = tid; e < (K / 64) * 512; e += kStKeyThreads) {
                const int blk_i = e >> 9, ee = e & 511;
                uint4 *p = reinterpret_cast<uint4 *>(sm + L::qbuf(n) + blk_i * 8192 + ee * 16);
                const float g = gam[ee >> 3];
                uint4 w = *p;
                uint32_t *wv = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float2 f =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[c]));
                    wv[c] = pack_bf16(f.x * g, f.y * g);
                }
                *p = w;
            }
            if (outs) {
                // P slot n % 2 was last read by O^T(n - 2) += U^T P^T: complete
                // with O^T(n - 1) += U^T P^T (bar_o2), which the state thread
                // issues only after key_ready(n - 1), so no later phase of
                // bar_o2 can have completed yet
                if (tid == 0 && n >= 1) ok = wait(&bar_o2, (n - 1) & 1);
                if (named_sync_or(kBarKey, kStKeyThreads, !ok)) { failed = true; break; }
                p_block_store(sm + L::ptile(n), pw[0], p_unit_i(warp), p_unit_j(warp), lane);
                if (pu2 >= 0) p_block_store(sm + L::ptile(n), pw[1], p_unit_i(pu2), p_unit_j(pu2), lane);
            }
            fence_proxy_async_smem();
            named_sync(kBarKey, kStKeyThreads);
            if (tid == 0) mbar_arrive(&key_ready[n & 3]);
            // this chunk's register slot takes chunk n + 2's gate inputs
            if (p2 == 0)
                prefetch_gates(n + 2, 0);
            else
                prefetch_gates(n + 2, 1);
        }
    } else if (tid < kKeyThreads) {
        // ================================================================ issuer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
        if (tid == kStIssuer) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (outs) tma_prefetch_desc(tm_out);
            // chunk n's k (q) boxes into K (Q) ring slot n % 3
            auto load_k = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                uint64_t *bar = &k_full[n % L::NK];
                mbar_arrive_expect_tx(bar, L::BOX);
                tma_load_4d(sm + L::kbuf(n), &tm_k, bar, 0, h, t0 + n * 64, b);
                if (K == 128) tma_load_4d(sm + L::kbuf(n) + 8192, &tm_k, bar, 64, h, t0 + n * 64, b);
            };
            auto load_q = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                uint64_t *bar = &q_full[n % L::NQ];
                mbar_arrive_expect_tx(bar, L::BOX);
                tma_load_4d(sm + L::qbuf(n), &tm_q, bar, 0, h, t0 + n * 64, b);
                if (K == 128) tma_load_4d(sm + L::qbuf(n) + 8192, &tm_q, bar, 64, h, t0 + n * 64, b);
            };
            auto load_v = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                uint64_t *bar = &v_full[n % L::NV];
                uint8_t *dst = sm + L::vbuf(n);
                mbar_arrive_expect_tx(bar, L::V_BYTES);
                tma_load_4d(dst, &tm_v, bar, 0, h, t0 + n * 64, b);
                tma_load_4d(dst + 8192, &tm_v, bar, 64, h, t0 + n * 64, b);
            };
            // chunk n's [T'^T | T''^T] into ring slot n % 2
            auto load_tt = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                mbar_arrive_expect_tx(&tt_full[n % L::NT], 16384);
                bulk_load(sm + L::tp(n), prep_seq + (size_t)n * kPrepChunkBytes + kPrepTP, 16384,
                          &tt_full[n % L::NT]);
            };
            // W^T(n) = K^T T'^T into the W^T columns
            auto issue_w = [&](int n) -> bool {
                if (!wait(&k_full[n % L::NK], (n / L::NK) & 1)) return false;
                if (!wait(&tt_full[n % L::NT], (n / L::NT) & 1)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tb + L::WT, sdesc(base + L::kbuf(n) + ks * 2048, 8192, 1024),
                             sdesc(base + L::tp(n) + ks * 2048, 8192, 1024), I_ABMN, ks > 0);
                mma_commit(&bar_w);
                return true;
            };
            // U~^T(n) = V^T T''^T into U slot n % 2 (none with v = 0)
            auto issue_ut = [&](int n) -> bool {
                if (zero_v) return true;
                if (!wait(&v_full[n % L::NV], (n / L::NV) & 1)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tb + L::ua(n), sdesc(base + L::vbuf(n) + ks * 2048, 8192, 1024),
                             sdesc(base + L::tpp(n) + ks * 2048, 8192, 1024), I_ABMN, ks > 0);
                mma_commit(&bar_ut);
                return true;
            };
            // launched as a programmatic dependent, this kernel may have started
            // before the key-side pass ended: its operands (and, in the
            // gathering form, q' and k') are read only after it
            pdl_wait();
            for (int m = 0; m < 2 && m < nchunks; ++m) {
                load_k(m);
                load_q(m);
                load_tt(m);
                if (!zero_v) load_v(m);
            }
            bool ok = issue_w(0) && issue_ut(0);
            for (int n = 0; ok && n < nchunks; ++n) {
                // ---- chunk n's window ----
                // the key group is done with chunk n (gamma Q(n) is in place),
                // and the state thread has issued U(n) (u_sig), after the state
                // group read W^T(n) out (its columns take W^T(n+1) below)
                ok = wait(&key_ready[n & 3], (n >> 2) & 1) && wait(&u_sig, n & 1);
                if (ok && outs) {
                    // O^T(n) = S(n-1) (gamma Q(n))^T.  O^T(n-2) has been read
                    // out: its store warps joined the state group's barrier at
                    // the top of chunk n - 1
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks) {
                        const uint32_t ko = (ks / 4) * 8192 + (ks % 4) * 32;
                        mma_bf16_ta(tb + L::ocol(n), tb + L::SBT + 8 * ks,
                                    sdesc(base + L::qbuf(n) + ko, 16, 1024), I_MM, ks > 0);
                    }
                    mma_commit(&bar_os);
                }
                // U(n) is complete, and with it dS(n - 1) and O^T(n - 1) += U^T P^T
                ok = ok && wait(&bar_u, n & 1);
                if (!ok) break;
                // chunk n + 2's loads first (they have the longest way to
                // go).  K and Q slot (n + 2) % 3 held chunk n - 1, read by
                // W^T(n - 1) and dS(n - 1) (bar_u(n) covers the state
                // thread's earlier products), the key group (done: key_ready)
                // and this thread's S-term of O^T(n - 1) (done: the state
                // thread waited for it before O^T(n - 1) += U^T P^T); the
                // [T'^T | T''^T] slot held chunk n, read by W^T(n) (seen by the
                // state group) and U~^T(n) (before U(n)); V(n) was read by U~^T(n)
                if (n + 2 < nchunks) {
                    load_k(n + 2);
                    load_q(n + 2);
                    load_tt(n + 2);
                    if (!zero_v) load_v(n + 2);
                }
                // the next chunk's W^T (the state group reads it out into the
                // -W^T tile while dS(n) runs) and U~^T, into U(n - 1)'s slot
                if (n + 1 < nchunks) ok = issue_w(n + 1) && issue_ut(n + 1);
            }
            if (!ok) failed = true;
        }
    } else {
        // ================================================================ state group
        asm volatile("setmaxnreg.inc.sync.aligned.u32 144;" ::: "memory");
        const int sid = tid - kKeyThreads;  // 0..255
        const int sw = sid >> 5;            // state warp 0..7
        const int c = quad_row;             // state row = TMEM lane = value channel
        const int hf = sw >> 2;             // column half
        // initial state: fp32 registers + bf16 operand copy in TMEM
        float S[KH];
        {
            const int j0 = hf * KH;
#pragma unroll
            for (int j = 0; j < KH; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tk.s0p) x = *reinterpret_cast<const float4 *>(tk.s0p + (size_t)c * K + j0 + j);
                if (tk.s0_identity) {
                    x.x = (c == j0 + j) ? 1.f : 0.f;
                    x.y = (c == j0 + j + 1) ? 1.f : 0.f;
                    x.z = (c == j0 + j + 2) ? 1.f : 0.f;
                    x.w = (c == j0 + j + 3) ? 1.f : 0.f;
                }
                S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
            }
#pragma unroll
            for (int p = 0; p < KH / 32; ++p) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = S[32 * p + i];
                uint32_t w[16];
                pack_row(v, w);
                tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        named_sync(kBarState, kStateThreads);

        // U^T = U~^T + S (-W^T) of chunk m (state thread), once the state
        // group has written -W^T and U~^T is complete; then u_sig tells the
        // issuer that U(m) is issued and S(m-1) in place for the S-term.
        auto issue_u = [&](int m) -> bool {
            if (!zero_v && !wait(&bar_ut, m & 1)) return false;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                // with v = 0 there is no U~ product: this one starts the accumulator
                mma_bf16_ta(tb + L::ua(m), tb + L::SBT + 8 * ks,
                            sdesc(base + L::NWB + ks * 2048, 8192, 1024), I_BMN,
                            zero_v ? (uint32_t)(ks > 0) : 1u);
            mma_commit(&bar_u);
            // the issuer's S-term of O^T(m) may read the bf16 S(m-1) now
            tc_fence_before();
            mbar_arrive(&u_sig);
            return true;
        };
        // chunk m's O^T -> the staging tile, by warps 12-15 (TMEM lane quarter
        // w % 4, all 64 columns), then a TMA store by warp 11.  Called by warps
        // 11-15; one thread waits for the products, warp 11 for the previous
        // store to have read the tile, and all 160 take the same branch on a
        // timeout (false).
        auto store_out = [&](int m) -> bool {
            bool okw = true;
            if (sid == 128) okw = wait(&bar_o2, m & 1);
            if (sw == 3 && lane == 0) bulk_wait_read_all();
            if (named_sync_or(kBarOut, 160, !okw)) return false;
            if (sw >= 4) {
                tc_fence_after();
                const bool odd = lane & 1;
                uint8_t *tile = sm + L::OST + (c >> 6) * 8192;
                const uint32_t cb = (uint32_t)(c & 63) >> 3, cw = (uint32_t)(c & 6) * 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    tmem_ld32(tb + lane_off + L::ocol(m) + 32 * half, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        // pairs of lanes swap one value: each writes two channels of one token
                        const float got = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[i + 1], 1);
                        const uint32_t t = 32 * half + i + (odd ? 1 : 0);
                        const float lo = odd ? got : v[i], hi = odd ? v[i + 1] : got;
                        *reinterpret_cast<uint32_t *>(tile + swz128(t, cb) + cw) =
                            pack_bf16(lo, hi);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
            }
            named_sync(kBarOut2, 160);  // the tile is written
            if (sw == 3 && lane == 0) {
                if (bounds_ok(m >= 0 && m < nchunks, status)) {
                    tma_store_4d(tm_out, sm + L::OST, 0, h, t0 + m * 64, b);
                    tma_store_4d(tm_out, sm + L::OST + 8192, 64, h, t0 + m * 64, b);
                }
                bulk_commit_group();
            }
            return true;
        };
        // -W^T(m) from TMEM into its operand tile: state warp sw reads TMEM
        // lane quarter sw % 4, column half sw / 4, once W^T(m) is complete
        // (U(m - 1), the reader of the previous -W^T, is complete too).  All
        // state threads take the same branch on a timeout (false).
        auto read_w = [&](int m) -> bool {
            bool okw = true;
            if (sid == 0) okw = wait(&bar_w, m & 1);
            if (named_sync_or(kBarState, kStateThreads, !okw)) return false;
            if (quad_row < K) {
                tc_fence_after();
                float v[32];
                tmem_ld32(tb + lane_off + L::WT + 32 * hf, v);
                tmem_ld_wait();
                store_row<4>(sm + L::NWB, quad_row, 4 * hf, v, -1.f);
            }
            // the tile feeds U(m); W^T's columns take W^T(m + 1) after u_sig(m)
            fence_proxy_async_smem();
            tc_fence_before();
            return true;
        };
        if (!read_w(0)) failed = true;
        named_sync(kBarState, kStateThreads);
        if (sw == 0 && !failed) {
            bool ok0 = true;
            if (lane == 0) ok0 = issue_u(0);
            ok0 = __shfl_sync(0xffffffffu, ok0, 0);
            failed = !ok0;
        }

        for (int n = 0; n < nchunks; ++n) {
            // ---- U epilogue: bf16 U^T and U^T diag(decay) into the U slot ----
            const float *slot = sg + (n % 3) * 68;
            float gC;  // read with the decays: the slot is rewritten for chunk n + 3
            bool ok = !failed;
            // U(n) complete; the key group's decays, P(n) and gamma Q(n) in place
            if (sid == 0 && ok) ok = wait(&bar_u, n & 1) && wait(&key_ready[n & 3], (n >> 2) & 1);
            if (named_sync_or(kBarState, kStateThreads, !ok)) { failed = true; break; }
            {
                tc_fence_after();
                // each thread rewrites only the 32 columns it has read
                gC = slot[64];
                float v[32];
                tmem_ld32(tb + lane_off + L::ua(n) + 32 * hf, v);
                tmem_ld_wait();
                uint32_t w[16];
                if (outs) {
                    pack_row(v, w);
                    tmem_st16(tb + lane_off + L::ua(n) + 32 * hf, w);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= slot[32 * hf + i];
                pack_row(v, w);
                tmem_st16(tb + lane_off + L::ua(n) + 32 * hf + 16, w);
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            // ---- dS = U^T diag(decay) K, then O^T += U^T P^T (warp 8) ----
            if (sid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ta(tb + L::DS, tb + L::ud_col(n, ks),
                                sdesc(base + L::kbuf(n) + ks * 2048, 8192, 1024), I_DS, ks > 0);
                mma_commit(&bar_s);
                if (outs) {
                    // after the issuer's S-term of O^T(n), which also reads
                    // S(n-1) (overwritten by the update below); P(n) is in
                    // place since key_ready(n), waited before the epilogue
                    ok = wait(&bar_os, n & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tb + L::ocol(n), tb + L::ut_col(n, ks),
                                        sdesc(base + L::ptile(n) + ks * 32, 16, 1024), I_MM, 1);
                        mma_commit(&bar_o2);
                    }
                }
            }
            // ---- -W^T(n+1) while dS(n) runs ----
            if (n + 1 < nchunks && !read_w(n + 1)) ok = false;
            if (sid == 0) ok = ok && wait(&bar_s, n & 1);
            if (named_sync_or(kBarState, kStateThreads, !ok)) { failed = true; break; }
            // ---- state update: S <- gamma_C S + dS, and its bf16 copy ----
            {
                tc_fence_after();
                const int j0 = hf * KH;
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
                    uint32_t w[16];
                    pack_row(v, w);
                    tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            // ---- next chunk's U (warp 8); this chunk's output (warps 11-15) ----
            bool ok1 = true;
            if (sw == 0) {
                if (lane == 0 && n + 1 < nchunks) ok1 = issue_u(n + 1);
                ok1 = __shfl_sync(0xffffffffu, ok1, 0);
            } else if (sw >= 3 && outs) {
                ok1 = store_out(n);
            }
            if (!ok1) failed = true;
        }
        if (sw == 3 && lane == 0 && outs) bulk_wait_all();  // outputs written before the CTA ends
        if (!failed && tk.stp != nullptr) {
            const int j0 = hf * KH;
#pragma unroll
            for (int j = 0; j < KH; j += 4)
                *reinterpret_cast<float4 *>(tk.stp + (size_t)c * K + j0 + j) =
                    make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    }

    if (failed) *abort_v = 1;
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        // products still in flight read shared memory and write TMEM: each
        // issuing thread's commit completes once all of its products have
        if (tid == kStIssuer || tid == kKeyThreads) {
            uint64_t *d = &drain[tid == kStIssuer ? 0 : 1];
            mma_commit(d);
            mbar_wait(d, 0, kSpinLimit / 16);
        }
        if (tid == kStIssuer) {
            if (status) atomicOr(status, kStatusTimeout);
            // let in-flight loads land before the CTA's shared memory is released
            uint64_t *loads[] = {&k_full[0], &k_full[1], &k_full[2], &q_full[0], &q_full[1],
                                 &q_full[2], &v_full[0], &v_full[1], &tt_full[0], &tt_full[1]};
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

// ---------------------------------------------------------------- one-pass (fused) kernel
// The one-pass form: one CTA per (b, h) sequence (or segment) computes the
// key-side operands of every chunk on chip and runs the state chain beside
// them, so no operand goes through global memory.  12 warps:
//   key group   (warps 0-3): gates, [K;Q] K^T on the tensor cores, A and P,
//               the inverse and T'^T, T''^T (above), then W^T and U~^T, the
//               -W^T operand over the spent T'^T / T''^T slot, and gamma
//               folded into the Q tile.  Thread 0 issues its products and
//               the q/k / V loads.  It depends on no state and runs up to two
//               chunks ahead of the state group: the T'/T'' (then -W^T), P,
//               U~ and V slots are per chunk parity, the q/k stages three.
//   state group (warps 4-11): the state chain of the two-pass state kernel
//               above, unchanged -- U, epilogue, dS, fp32 update, and the
//               transposed output staged for TMA stores by warps 7-11.
// The key group's [K;Q] K^T and W^T share 64 TMEM columns (one is read out
// before the other is written), which leaves room for two output
// accumulators.  Handoffs: nw_ready (key -> state: -W^T, U~^T, P, gamma Q
// and the chunk's decays are in place), tt_free (U has read -W^T: the slot
// takes chunk n + 2's T'^T, T''^T), uap_free (the U slot and P are spent).
template <int K>
struct FuLayout {
    static constexpr int NSTAGE = 3;
    // q/k stage: the K and Q boxes of one 64-channel block adjacent, so that
    // [K;Q] is one 128-row operand; the K blocks KLBO bytes apart
    static constexpr uint32_t KC0 = 0, QC0 = 8192, KC1 = 16384, QC1 = 24576;
    static constexpr uint32_t STAGE = K == 128 ? 32768 : 16384;
    static constexpr uint32_t KLBO = K == 128 ? 16384 : 8192;
    static constexpr uint32_t VB = NSTAGE * STAGE;            // V ring, two 16 KB slots
    static constexpr uint32_t TT = VB + 2 * 16384;            // [T'^T | T''^T] / -W^T, two slots
    static constexpr uint32_t PP = TT + 2 * 16384;            // P, two 8 KB slots
    static constexpr uint32_t OST = PP + 2 * 8192;            // output staging, 2 x 64 x 64
    static constexpr uint32_t AF = OST + 16384;               // float [64][68]
    static constexpr uint32_t KGATE = AF + 64 * kLD * 4;      // G2, gamma, beta
    static constexpr uint32_t SGATE = KGATE + 3 * 64 * 4;     // 3 x (decay[64], gamma_C)
    static constexpr uint32_t END = SGATE + 3 * 68 * 4;
    static constexpr uint32_t KQ_BYTES = (K == 128 ? 4u : 2u) * 8192u;
    static constexpr uint32_t V_BYTES = 2u * 8192u;
    static constexpr size_t SMEM = END;
    static_assert(SMEM + 1024 <= 232448, "shared memory budget");
    static __device__ __forceinline__ uint32_t tp(int n) { return TT + (n & 1) * 16384; }
    static __device__ __forceinline__ uint32_t tpp(int n) { return tp(n) + 8192; }
    static __device__ __forceinline__ uint32_t nw(int n) { return tp(n); }
    static __device__ __forceinline__ uint32_t ptile(int n) { return PP + (n & 1) * 8192; }
    static __device__ __forceinline__ uint32_t vbuf(int n) { return VB + (n & 1) * 16384; }
    // TMEM columns: [K;Q] K^T / W^T, U~^T / U^T of even / odd chunks, O^T of
    // even / odd chunks, the bf16 state, dS
    static constexpr uint32_t KW = 0, UA = 64, O0 = 192, O1 = 256, SBT = 320, DS = 384;
    static __device__ __forceinline__ uint32_t ocol(int n) { return (n & 1) ? O1 : O0; }
    static __device__ __forceinline__ uint32_t ua(int n) { return UA + 64 * (n & 1); }
    static __device__ __forceinline__ uint32_t ut_col(int n, int ks) {
        return ua(n) + 32 * (ks >> 1) + 8 * (ks & 1);
    }
    static __device__ __forceinline__ uint32_t ud_col(int n, int ks) { return ut_col(n, ks) + 16; }
};

constexpr int kFuKeyThreads = 128;
constexpr int kFuThreads = kFuKeyThreads + kStateThreads;

template <int K>
__global__ void __launch_bounds__(kFuThreads, 1)
    prefill_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ alpha,
                         const float *__restrict__ beta, const float *__restrict__ S0,
                         bool want_o, float *__restrict__ ST, int T, int Ts, int H, int BH,
                         SegPlan plan, int *status) {
    using L = FuLayout<K>;
    constexpr int KH = K / 2;  // state columns per state-group thread
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && status) atomicOr(status, kStatusBounds);
        return;
    }
    uint8_t *sm = smem_raw;
    __shared__ uint64_t kq_full[3], v_full[2], bar_kq, bar_w, bar_u, bar_s, bar_o2, nw_ready[2],
        tt_free[2], uap_free[2], drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int *abort_v = &abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const SegTask tk = segment_task(plan, K, T, S0, ST, BH);
    // (every thread takes the same branch, before any barrier or allocation)
    if (!bounds_ok(tk.seq < (size_t)BH && tk.t0 >= 0 && tk.t0 < tk.t1 && tk.t1 <= T &&
                       tk.t0 % 64 == 0 && T <= Ts,
                   status))
        return;
    const size_t seq = tk.seq;
    const int t0 = tk.t0, t1 = tk.t1;
    const bool zero_v = tk.zero_v;
    const bool outs = want_o && tk.outputs;
    const int b = (int)(seq / H), h = (int)(seq % H);
    const int nchunks = (t1 - t0 + 63) / 64;
    const uint32_t base = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (outs) tma_prefetch_desc(&tm_o);
        uint64_t *bars[] = {&kq_full[0], &kq_full[1], &kq_full[2], &v_full[0],   &v_full[1],
                            &bar_kq,     &bar_w,      &bar_u,      &bar_s,       &bar_o2,
                            &nw_ready[0], &nw_ready[1], &tt_free[0], &tt_free[1], &uap_free[0],
                            &uap_free[1], &drain[0],  &drain[1]};
        for (uint64_t *bb : bars) mbar_init(bb, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int quad_row = (warp & 3) * 32 + lane;  // TMEM lane of this thread
    // decay[64] and gamma_C of chunk n in slot n % 3 (written by the key group)
    float *sg = reinterpret_cast<float *>(sm + L::SGATE);

    auto load_kq = [&](int n) {
        if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
        const int st = n % L::NSTAGE;
        uint8_t *stg = sm + st * L::STAGE;
        mbar_arrive_expect_tx(&kq_full[st], L::KQ_BYTES);
        tma_load_4d(stg + L::KC0, &tm_k, &kq_full[st], 0, h, t0 + n * 64, b);
        tma_load_4d(stg + L::QC0, &tm_q, &kq_full[st], 0, h, t0 + n * 64, b);
        if (K == 128) {
            tma_load_4d(stg + L::KC1, &tm_k, &kq_full[st], 64, h, t0 + n * 64, b);
            tma_load_4d(stg + L::QC1, &tm_q, &kq_full[st], 64, h, t0 + n * 64, b);
        }
    };
    auto load_v = [&](int n) {
        if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
        uint64_t *bar = &v_full[n & 1];
        uint8_t *dst = sm + L::vbuf(n);
        mbar_arrive_expect_tx(bar, L::V_BYTES);
        tma_load_4d(dst, &tm_v, bar, 0, h, t0 + n * 64, b);
        tma_load_4d(dst + 8192, &tm_v, bar, 64, h, t0 + n * 64, b);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_or_abort(bar, parity, kSpinLimit, abort_v);
        if (!ok) *abort_v = 1;
        return ok;
    };

    constexpr uint32_t I_MM = idesc_bf16(128, 64, false, false);  // K-major x K-major, N = 64
    constexpr uint32_t I_ABMN = idesc_bf16(128, 64, true, true);  // MN-major A and B
    constexpr uint32_t I_BMN = idesc_bf16(128, 64, false, true);  // MN-major B, N = 64
    constexpr uint32_t I_DS = idesc_bf16(128, K, false, true);    // MN-major B, N = K

    bool failed = false;

    if (tid < kFuKeyThreads) {
        // ================================================================ key group
        float *AF = reinterpret_cast<float *>(sm + L::AF);
        float *G2 = reinterpret_cast<float *>(sm + L::KGATE);
        float *gam = G2 + 64;
        float *bet = G2 + 128;
        float pa0 = 1.f, pa1 = 1.f, pb0 = 0.f, pb1 = 0.f;  // prefetched gate inputs (warp 1)
        auto prefetch_gates = [&](int n) {
            if (warp == 1 && n < nchunks) {
                const int nv = min(64, t1 - t0 - n * 64);
                const size_t i0 = ((size_t)b * Ts + t0 + n * 64 + lane) * H + h;
                const size_t i1 = i0 + (size_t)32 * H;
                pa0 = lane < nv ? alpha[i0] : 1.f;
                pb0 = lane < nv ? beta[i0] : 0.f;
                pa1 = lane + 32 < nv ? alpha[i1] : 1.f;
                pb1 = lane + 32 < nv ? beta[i1] : 0.f;
            }
        };
        prefetch_gates(0);
        if (tid == 0) {
            for (int m = 0; m < L::NSTAGE && m < nchunks; ++m) load_kq(m);
            if (!zero_v)
                for (int m = 0; m < 2 && m < nchunks; ++m) load_v(m);
        }
        for (int n = 0; n < nchunks; ++n) {
            const int st = n % L::NSTAGE;  // q/k stage
            const int p2 = n & 1;          // ring slots of this chunk
            const uint32_t stg = base + st * L::STAGE;
            const int nvalid = min(64, t1 - t0 - n * 64);
            bool ok = true;
            if (tid == 0) {
                ok = wait(&kq_full[st], (n / L::NSTAGE) & 1);
                if (ok) {
                    tc_fence_after();
                    issue_kq_kt<K>(tb + L::KW, stg, L::KC0, L::KC1);
                    mma_commit(&bar_kq);
                }
                // chunk n - 2 is done with this parity's slots: U has read its
                // -W^T (T'/T'' slot), and dS and O^T += U^T P^T have read its U
                // slot and P
                if (ok && n >= 2) ok = wait(&tt_free[p2], ((n - 2) >> 1) & 1);
                if (ok && n >= 2) ok = wait(&uap_free[p2], ((n - 2) >> 1) & 1);
                if (ok) ok = wait(&bar_kq, n & 1);
            }
            if (warp == 1) {
                chunk_gates(pa0, pa1, pb0, pb1, lane, nvalid, G2, gam, bet);
                __syncwarp();
                // the state group's decay to the chunk end and gamma_C; slot
                // n % 3 was last read in the state epilogue of chunk n - 3,
                // which precedes the uap_free of chunk n - 3 waited for above
                // (in the previous iteration)
                float *slot = sg + (n % 3) * 68;
                const float gC = G2[63];
                slot[lane] = exp2f(gC - G2[lane]);
                slot[lane + 32] = exp2f(gC - G2[lane + 32]);
                if (lane == 0) slot[64] = exp2f(gC);
            }
            if (named_sync_or(kBarKey, kFuKeyThreads, !ok)) { failed = true; break; }

            // ---- A (fp32, solve input) and P (bf16 operand) ----
            tc_fence_after();
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch)
                chunk_ap(tb + lane_off + L::KW + 32 * ch, quad_row, ch, G2, bet, AF,
                         outs ? sm + L::ptile(n) : nullptr);
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarKey, kFuKeyThreads);
            // ---- T = (I + A)^{-1}; T'^T, T''^T ----
            chunk_inverse_tprime<kFuKeyThreads>(AF, bet, gam, sm + L::tp(n), sm + L::tpp(n), tid);
            fence_proxy_async_smem();
            named_sync(kBarKey, kFuKeyThreads);

            // ---- W^T = K^T T'^T and U~^T = V^T T''^T ----
            if (tid == 0) {
                if (!zero_v) ok = wait(&v_full[p2], (n >> 1) & 1);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        mma_bf16(tb + L::KW, sdesc(stg + L::KC0 + ks * 2048, L::KLBO, 1024),
                                 sdesc(base + L::tp(n) + ks * 2048, 8192, 1024), I_ABMN, ks > 0);
                        if (!zero_v)
                            mma_bf16(tb + L::ua(n), sdesc(base + L::vbuf(n) + ks * 2048, 8192, 1024),
                                     sdesc(base + L::tpp(n) + ks * 2048, 8192, 1024), I_ABMN,
                                     ks > 0);
                    }
                    mma_commit(&bar_w);
                }
            }
            {
                // Q <- diag(gamma) Q in place while the products run (they read
                // the K blocks, V and T'^T, T''^T; Q is next read by O^T)
                uint8_t *stq = sm + st * L::STAGE;
#pragma unroll
                for (int e = tid; e < (K / 64) * 512; e += kFuKeyThreads) {
                    const int blk_i = e >> 9, ee = e & 511;
                    uint4 *p = reinterpret_cast<uint4 *>(stq + (blk_i ? L::QC1 : L::QC0) + ee * 16);
                    const float gq = gam[ee >> 3];
                    uint4 w = *p;
                    uint32_t *wv = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float2 f =
                            __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[c]));
                        wv[c] = pack_bf16(f.x * gq, f.y * gq);
                    }
                    *p = w;
                }
            }
            if (tid == 0 && ok) {
                ok = wait(&bar_w, n & 1);
                // U~^T has read this V slot
                if (ok && !zero_v && n + 2 < nchunks) load_v(n + 2);
            }
            if (named_sync_or(kBarKey, kFuKeyThreads, !ok)) { failed = true; break; }
            {
                // -W^T over T'^T, T''^T (consumed by the products above)
                tc_fence_after();
                if (quad_row < K) {
#pragma unroll 1
                    for (int ch = 0; ch < 2; ++ch) {
                        float v[32];
                        tmem_ld32(tb + lane_off + L::KW + 32 * ch, v);
                        tmem_ld_wait();
                        store_row<4>(sm + L::nw(n), quad_row, 4 * ch, v, -1.f);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (named_sync_or(kBarKey, kFuKeyThreads, !ok)) { failed = true; break; }
            if (tid == 0) mbar_arrive(&nw_ready[p2]);
            prefetch_gates(n + 1);
        }
    } else {
        // ================================================================ state group
        const int sid = tid - kFuKeyThreads;  // 0..255
        const int sw = sid >> 5;              // state warp 0..7
        const int c = quad_row;               // state row = TMEM lane = value channel
        const int hf = sw >> 2;               // column half
        // initial state: fp32 registers + bf16 operand copy in TMEM
        float S[KH];
        {
            const int j0 = hf * KH;
#pragma unroll
            for (int j = 0; j < KH; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tk.s0p) x = *reinterpret_cast<const float4 *>(tk.s0p + (size_t)c * K + j0 + j);
                if (tk.s0_identity) {
                    x.x = (c == j0 + j) ? 1.f : 0.f;
                    x.y = (c == j0 + j + 1) ? 1.f : 0.f;
                    x.z = (c == j0 + j + 2) ? 1.f : 0.f;
                    x.w = (c == j0 + j + 3) ? 1.f : 0.f;
                }
                S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
            }
#pragma unroll
            for (int p = 0; p < KH / 32; ++p) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = S[32 * p + i];
                uint32_t w[16];
                pack_row(v, w);
                tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        named_sync(kBarState, kStateThreads);

        // U^T += S (-W^T) of chunk m, then O^T = S (gamma Q)^T (warp 4, once
        // the key group handed chunk m over)
        auto issue_u = [&](int m) -> bool {
            if (!wait(&nw_ready[m & 1], (m >> 1) & 1)) return false;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                // with v = 0 there is no U~ product: this one starts the accumulator
                mma_bf16_ta(tb + L::ua(m), tb + L::SBT + 8 * ks,
                            sdesc(base + L::nw(m) + ks * 2048, 8192, 1024), I_BMN,
                            zero_v ? (uint32_t)(ks > 0) : 1u);
            mma_commit(&bar_u);
            if (outs) {
                const uint32_t stg = base + (m % L::NSTAGE) * L::STAGE;
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const uint32_t kb = ks / 4, ko = (ks % 4) * 32;
                    mma_bf16_ta(tb + L::ocol(m), tb + L::SBT + 8 * ks,
                                sdesc(stg + (kb ? L::QC1 : L::QC0) + ko, 16, 1024), I_MM, ks > 0);
                }
            }
            return true;
        };
        // chunk m's O^T -> the staging tile, by warps 8-11 (TMEM lane quarter
        // w % 4, all 64 columns), then a TMA store by warp 7.  Called by warps
        // 7-11; one thread waits for the products, warp 7 for the previous
        // store to have read the tile, and all 160 take the same branch on a
        // timeout (false).
        auto store_out = [&](int m) -> bool {
            bool okw = true;
            if (sid == 128) okw = wait(&bar_o2, m & 1);
            if (sw == 3 && lane == 0) bulk_wait_read_all();
            if (named_sync_or(kBarOut, 160, !okw)) return false;
            if (sw >= 4) {
                tc_fence_after();
                const bool odd = lane & 1;
                uint8_t *tile = sm + L::OST + (c >> 6) * 8192;
                const uint32_t cb = (uint32_t)(c & 63) >> 3, cw = (uint32_t)(c & 6) * 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    tmem_ld32(tb + lane_off + L::ocol(m) + 32 * half, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        // pairs of lanes swap one value: each writes two channels of one token
                        const float got = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[i + 1], 1);
                        const uint32_t t = 32 * half + i + (odd ? 1 : 0);
                        const float lo = odd ? got : v[i], hi = odd ? v[i + 1] : got;
                        *reinterpret_cast<uint32_t *>(tile + swz128(t, cb) + cw) =
                            pack_bf16(lo, hi);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
            }
            named_sync(kBarOut2, 160);  // the tile is written
            if (sw == 3 && lane == 0) {
                if (bounds_ok(m >= 0 && m < nchunks, status)) {
                    tma_store_4d(&tm_o, sm + L::OST, 0, h, t0 + m * 64, b);
                    tma_store_4d(&tm_o, sm + L::OST + 8192, 64, h, t0 + m * 64, b);
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
            const int st = n % L::NSTAGE;
            const int p2 = n & 1;
            const uint32_t stg = base + st * L::STAGE;
            // ---- U epilogue: bf16 U^T and U^T diag(decay) into the U slot ----
            const float *slot = sg + (n % 3) * 68;
            float gC;  // read with the decays: the slot is rewritten for chunk n + 3
            bool ok = !failed;
            if (sid == 0 && ok) {
                ok = wait(&bar_u, n & 1);
                // U^T has read -W^T: the slot takes chunk n + 2's T'^T, T''^T
                if (ok) mbar_arrive(&tt_free[p2]);
            }
            if (named_sync_or(kBarState, kStateThreads, !ok)) { failed = true; break; }
            {
                tc_fence_after();
                // each thread rewrites only the 32 columns it has read
                gC = slot[64];
                float v[32];
                tmem_ld32(tb + lane_off + L::ua(n) + 32 * hf, v);
                tmem_ld_wait();
                uint32_t w[16];
                if (outs) {
                    pack_row(v, w);
                    tmem_st16(tb + lane_off + L::ua(n) + 32 * hf, w);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= slot[32 * hf + i];
                pack_row(v, w);
                tmem_st16(tb + lane_off + L::ua(n) + 32 * hf + 16, w);
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            // ---- dS = U^T diag(decay) K, then O^T += U^T P^T (warp 4) ----
            if (sid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ta(tb + L::DS, tb + L::ud_col(n, ks),
                                sdesc(stg + L::KC0 + ks * 2048, L::KLBO, 1024), I_DS, ks > 0);
                mma_commit(&bar_s);
                if (outs) {
                    // P of chunk n was written before its nw_ready
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ta(tb + L::ocol(n), tb + L::ut_col(n, ks),
                                    sdesc(base + L::ptile(n) + ks * 32, 16, 1024), I_MM, 1);
                    mma_commit(&bar_o2);
                }
                ok = wait(&bar_s, n & 1);
                if (ok) {
                    // dS(n) and, before it, O^T's first product have read q/k
                    // stage n % 3 (the key group is done with it): chunk n + 3
                    if (n + L::NSTAGE < nchunks) load_kq(n + L::NSTAGE);
                    if (!outs) mbar_arrive(&uap_free[p2]);  // dS has read the U slot
                }
            }
            if (named_sync_or(kBarState, kStateThreads, !ok)) { failed = true; break; }
            // ---- state update: S <- gamma_C S + dS, and its bf16 copy ----
            {
                tc_fence_after();
                const int j0 = hf * KH;
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
                    uint32_t w[16];
                    pack_row(v, w);
                    tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            // ---- next chunk's products (warp 4), releases (warp 6), this
            // ---- chunk's output (warps 7-11) ----
            bool ok1 = true;
            if (sw == 0) {
                if (lane == 0 && n + 1 < nchunks) ok1 = issue_u(n + 1);
            } else if (sw == 2) {
                // O^T += U^T P^T has completed (after dS, issued before it):
                // the U slot and P slot of this parity are free
                if (lane == 0 && outs) {
                    ok1 = wait(&bar_o2, n & 1);
                    if (ok1) mbar_arrive(&uap_free[p2]);
                }
            } else if (sw >= 3 && outs) {
                ok1 = store_out(n);
            }
            if (sw <= 2) ok1 = __shfl_sync(0xffffffffu, ok1, 0);
            if (!ok1) failed = true;
        }
        if (sw == 3 && lane == 0 && outs) bulk_wait_all();  // outputs written before the CTA ends
        if (!failed && tk.stp != nullptr) {
            const int j0 = hf * KH;
#pragma unroll
            for (int j = 0; j < KH; j += 4)
                *reinterpret_cast<float4 *>(tk.stp + (size_t)c * K + j0 + j) =
                    make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    }

    if (failed) *abort_v = 1;
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        // products still in flight read shared memory and write TMEM: each
        // issuing thread's commit completes once all of its products have
        if (tid == 0 || tid == kFuKeyThreads) {
            uint64_t *d = &drain[tid == 0 ? 0 : 1];
            mma_commit(d);
            mbar_wait(d, 0, kSpinLimit / 16);
        }
        if (tid == 0) {
            if (status) atomicOr(status, kStatusTimeout);
            // let in-flight loads land before the CTA's shared memory is released
            for (int s = 0; s < 3; ++s) {
                mbar_wait(&kq_full[s], 0, kSpinLimit / 16);
                mbar_wait(&kq_full[s], 1, kSpinLimit / 16);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_wait(&v_full[s], 0, kSpinLimit / 16);
                mbar_wait(&v_full[s], 1, kSpinLimit / 16);
            }
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

}  // namespace

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

// [B, Ts, H, C] bf16 tensor whose first T tokens per batch entry are used,
// viewed as 4-D (C, H, T, B) with 64 x 1 x 64 x 1 boxes.
bool make_token_map(CUtensorMap *m, const void *ptr, int B, int T, int Ts, int H, int C) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)C * 2 * H,
                             (cuuint64_t)C * 2 * H * Ts};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

namespace {

// Start states of the later segments: S_1 = E (end of segment 0) and
// S_{p+1} = S_p M_p + H_p, in float32 (with ST: one step more, the end
// state).  Rows of the state are independent, so a CTA owns 16 rows of one
// sequence; thread (j, g) = (tid % K, tid / K) holds column j of rows
// g RP .. g RP + RP - 1 (RP = K / 16).  Each step's M_p is staged in shared
// memory by coalesced 16-byte copies (the next step's while this one
// computes); the product reads one M element per row group and the 16 rows'
// entries of column m as broadcast float4 reads of a transposed copy.
template <int K>
struct CombineLayout {
    static constexpr size_t ST = 0;                              // rows^T [K][16] float
    static constexpr size_t MS = (size_t)K * 16 * 4;             // two [K][K] float buffers
    static constexpr size_t SMEM = MS + 2 * (size_t)K * K * 4;
};
template <int K>
__global__ void __launch_bounds__(256) segment_combine_kernel(float *ws, int BH, int nseg,
                                                              float *ST) {
    using L = CombineLayout<K>;
    constexpr int V = 128;
    constexpr int RP = K / 16;  // rows per thread
    static_assert(256 / K * RP == 16 && RP % 4 == 0, "combine thread mapping");
    extern __shared__ __align__(16) uint8_t smem_cb[];
    float *rowt = reinterpret_cast<float *>(smem_cb + L::ST);  // [m][row of the CTA]
    float *ms = reinterpret_cast<float *>(smem_cb + L::MS);
    const size_t VK = (size_t)V * K;
    const size_t seq = blockIdx.x;
    const int r0 = blockIdx.y * 16;
    const int tid = threadIdx.x;
    const int j = tid % K, g = tid / K;
    auto slot = [&](int kind, int p) { return ws + ((kind * (size_t)BH + seq) * nseg + p) * VK; };
    // M_p into buffer p % 2: K * K / 4 pieces of 16 bytes, cp.async (L2 only)
    auto stage = [&](int p) {
        const float *M = slot(1, p);
        float *dst = ms + (size_t)(p & 1) * K * K;
        for (int e = tid; e < K * K / 4; e += 256)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + 4 * e)),
                         "l"(M + 4 * e)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    const int last = ST != nullptr ? nseg : nseg - 1;  // steps p = 1 .. last - 1
    if (1 < last) stage(1);
    // element (row r0 + g RP + i, column j) of a V x K slot
    auto at = [&](int i) { return (size_t)(r0 + g * RP + i) * K + j; };
    float sv[RP];
    const float *E = slot(0, 0);
#pragma unroll
    for (int i = 0; i < RP; ++i) sv[i] = E[at(i)];
    for (int p = 1; p < nseg; ++p) {
        float *Sp = slot(2, p);
#pragma unroll
        for (int i = 0; i < RP; ++i) Sp[at(i)] = sv[i];
        if (p >= last) break;
        __syncthreads();  // every read of the previous rows and of buffer (p + 1) % 2 done
#pragma unroll
        for (int i = 0; i < RP; i += 4)
            *reinterpret_cast<float4 *>(rowt + j * 16 + g * RP + i) =
                make_float4(sv[i], sv[i + 1], sv[i + 2], sv[i + 3]);
        if (p + 1 < last) {
            stage(p + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // M_p and the rows in place
        const float *Ms = ms + (size_t)(p & 1) * K * K;
        const float *Hp = slot(0, p);
        float acc[RP];
#pragma unroll
        for (int i = 0; i < RP; ++i) acc[i] = Hp[at(i)];
#pragma unroll 4
        for (int m = 0; m < K; ++m) {
            const float mv = Ms[(size_t)m * K + j];
#pragma unroll
            for (int i = 0; i < RP; i += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(rowt + m * 16 + g * RP + i);
                acc[i] = fmaf(x.x, mv, acc[i]);
                acc[i + 1] = fmaf(x.y, mv, acc[i + 1]);
                acc[i + 2] = fmaf(x.z, mv, acc[i + 2]);
                acc[i + 3] = fmaf(x.w, mv, acc[i + 3]);
            }
        }
#pragma unroll
        for (int i = 0; i < RP; ++i) sv[i] = acc[i];
    }
    if (ST != nullptr) {
#pragma unroll
        for (int i = 0; i < RP; ++i) ST[seq * VK + at(i)] = sv[i];
    }
}

// The outputs of segments p >= 1 from their start states (kFirstX):
// o_t <- o0_t + S_p x_t, for the tokens of segment p, with o0 (bf16, written
// by the zero-start run) in o and x (bf16, the first K of 128 channels,
// written by the identity-start run) in X.  S_p enters the products as bf16,
// as the state does in the state pass's own output products.  One CTA per
// (sequence, segment, split) walks 64-token tiles: S_p stays in shared
// memory, x tiles feed warp-level MMAs (m16n8k16, fp32 accumulation), each
// result is added to o0 in a shared-memory tile that is then written back
// in whole 16-byte pieces of o's rows.  The next tile's x and o0 load
// (cp.async) while this tile's products run; two CTAs share an SM.
constexpr int kCorrThreads = 256;
template <int K>
struct CorrLayout {
    static constexpr int LDB = K + 8;                        // bf16 row stride of S, x tiles
    static constexpr int LDO = 128 + 8;                      // bf16 row stride of the o tile
    static constexpr size_t SB = 0;                          // S_p [128][LDB]
    static constexpr size_t XT = SB + 128 * LDB * 2;         // two x tiles [64][LDB]
    static constexpr size_t OT = XT + 2 * 64 * LDB * 2;      // two o0 -> o tiles [64][LDO]
    static constexpr size_t SMEM = OT + 2 * 64 * LDO * 2;
};
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
template <int K>
__global__ void __launch_bounds__(kCorrThreads, 2)
    segment_correct_kernel(const float *__restrict__ ws, const __nv_bfloat16 *__restrict__ X,
                           __nv_bfloat16 *o, int T, int Ts, int H, int BH, int nseg, int seg_len,
                           int *status) {
    using L = CorrLayout<K>;
    constexpr int V = 128;
    extern __shared__ __align__(16) uint8_t smem_c[];
    __nv_bfloat16 *sb = reinterpret_cast<__nv_bfloat16 *>(smem_c + L::SB);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long seq = blockIdx.x;
    const int p = (int)blockIdx.y + 1;
    if (!bounds_ok(seq < BH && p < nseg && T <= Ts, status)) return;
    const int b = (int)(seq / H), h = (int)(seq % H);
    const size_t VK = (size_t)V * K;
    const int tb0 = p * seg_len, tb1 = min(T, tb0 + seg_len);
    const int ntile = (tb1 - tb0 + 63) / 64;
    // x buffer of the CTA's it-th tile
    auto xtile = [&](int it) {
        return reinterpret_cast<__nv_bfloat16 *>(smem_c + L::XT) + (it & 1) * 64 * L::LDB;
    };
    // x rows of a tile (zeros past the segment's end) into buffer it % 2
    auto load_x = [&](int tile, int it) {
        const int t0 = tb0 + 64 * tile, nt = min(64, tb1 - t0);
        __nv_bfloat16 *xt = xtile(it);
        for (int e = tid; e < 64 * (K / 8); e += kCorrThreads) {
            const int r = e / (K / 8), c8 = e % (K / 8);
            const int rr = r < nt ? r : 0;
            cp_async16(xt + r * L::LDB + 8 * c8,
                       X + (((size_t)b * T + t0 + rr) * H + h) * V + 8 * c8, r < nt);
        }
        cp_async_commit();
    };
    // o buffer of the CTA's it-th tile
    auto otile = [&](int it) {
        return reinterpret_cast<__nv_bfloat16 *>(smem_c + L::OT) + (it & 1) * 64 * L::LDO;
    };
    auto load_o = [&](int tile, int it) {
        const int t0 = tb0 + 64 * tile, nt = min(64, tb1 - t0);
        __nv_bfloat16 *ot = otile(it);
        for (int e = tid; e < 64 * (V / 8); e += kCorrThreads) {
            const int r = e / (V / 8), c8 = e % (V / 8);
            const int rr = r < nt ? r : 0;
            cp_async16(ot + r * L::LDO + 8 * c8,
                       o + (((size_t)b * Ts + t0 + rr) * H + h) * V + 8 * c8, r < nt);
        }
        cp_async_commit();
    };
    const int tile0 = (int)blockIdx.z;
    if (tile0 < ntile) {
        load_x(tile0, 0);
        load_o(tile0, 0);
    }
    const float *Sp = ws + ((2 * (size_t)BH + seq) * nseg + p) * VK;  // slot S of (seq, p)
    for (int e = tid; e < V * K / 4; e += kCorrThreads) {
        const float4 f = reinterpret_cast<const float4 *>(Sp)[e];
        const int r = (4 * e) / K, c = (4 * e) % K;
        uint2 w;
        w.x = pack_bf16(f.x, f.y);
        w.y = pack_bf16(f.z, f.w);
        *reinterpret_cast<uint2 *>(sb + r * L::LDB + c) = w;
    }
    const int mb = warp & 3, nh = warp >> 2;  // tokens 16 mb.., values 64 nh..
    const int g = lane >> 2, t4 = lane & 3;
    for (int tile = tile0, it = 0; tile < ntile; tile += (int)gridDim.z, ++it) {
        const int t0 = tb0 + 64 * tile, nt = min(64, tb1 - t0);
        // the previous tile's products and write-back are done with buffers
        // (it + 1) % 2
        __syncthreads();
        const bool more = tile + (int)gridDim.z < ntile;
        if (more) {
            load_x(tile + (int)gridDim.z, it + 1);
            load_o(tile + (int)gridDim.z, it + 1);
        }
        // this tile's x and o0: every group but the next tile's two
        if (more) cp_async_wait<2>(); else cp_async_wait<0>();
        __syncthreads();
        const __nv_bfloat16 *xt = xtile(it);
        __nv_bfloat16 *ot = otile(it);
        float d[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, smem_u32(xt + (16 * mb + (lane & 7) + 8 * ((lane >> 3) & 1)) * L::LDB +
                                16 * ks + 8 * (lane >> 4)));
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) {  // n-tiles 2 jp, 2 jp + 1
                const int mi = lane >> 3;
                const int row = 64 * nh + 8 * (2 * jp + (mi >> 1)) + (lane & 7);
                uint32_t bb[4];
                ldsm_x4(bb, smem_u32(sb + row * L::LDB + 16 * ks + 8 * (mi & 1)));
                mma_16816(d[2 * jp], a, bb[0], bb[1]);
                mma_16816(d[2 * jp + 1], a, bb[2], bb[3]);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = 64 * nh + 8 * j + 2 * t4;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                uint32_t *pr = reinterpret_cast<uint32_t *>(ot + (16 * mb + g + 8 * hr) * L::LDO + col);
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pr));
                *pr = pack_bf16(f.x + d[j][2 * hr], f.y + d[j][2 * hr + 1]);
            }
        }
        __syncthreads();
        for (int e = tid; e < 64 * (V / 8); e += kCorrThreads) {
            const int r = e / (V / 8), c8 = e % (V / 8);
            if (r < nt)
                reinterpret_cast<uint4 *>(o + (((size_t)b * Ts + t0 + r) * H + h) * V)[c8] =
                    *reinterpret_cast<const uint4 *>(ot + r * L::LDO + 8 * c8);
        }
    }
    cp_async_wait<0>();
}

template <int K, bool GATHER = false>
cudaError_t launch_prep(const CUtensorMap &mq, const CUtensorMap &mk, const float *alpha,
                        const float *beta, uint8_t *prep, long long BH, int T, int Ts, int H,
                        cudaStream_t stream, PrepGather gth = PrepGather{nullptr, nullptr, nullptr}) {
    auto kern = prefill_prep_kernel<K, GATHER>;
    using L = PrepLayout<K, GATHER>;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] != context_key()) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)L::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    // persistent CTAs, prep_ctas_per_sm per SM (the loop is correct for any residency)
    const long long total = BH * ((T + 63) / 64);
    const long long grid =
        std::min<long long>(total, (long long)prep_ctas_per_sm(GATHER) * sm_count());
    kern<<<(unsigned)grid, kPrepThreads, L::SMEM, stream>>>(mq, mk, alpha, beta, prep, T, Ts, H,
                                                           total, gth, device_status_ptr());
    return cudaGetLastError();
}

// Whole-sequence launch, or the segment-parallel sequence (first pass,
// combine, second pass) of the one-pass kernel (prep == nullptr) or of the
// state-side kernel of the two-pass form.  The two-pass form with an X
// buffer (xbuf, tensor map mx) replaces the second pass: the first pass
// writes every segment's o0 and X, the combine the end state, and
// segment_correct_kernel adds S_p x_t; without outputs it needs neither.
template <int K>
cudaError_t run_tc(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                   const CUtensorMap &mo, const float *alpha, const float *beta, const float *S0,
                   void *o, float *ST, long long BH, int T, int Ts, int H, const SegShape &sh,
                   float *ws, const uint8_t *prep, cudaStream_t stream,
                   const CUtensorMap *mx = nullptr, const __nv_bfloat16 *xbuf = nullptr) {
    static uintptr_t attr_set[2][64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int two = prep != nullptr;
    const size_t smem = two ? StLayout<K>::SMEM : FuLayout<K>::SMEM;
    if (attr_set[two][dev] != context_key()) {
        const cudaError_t e =
            two ? cudaFuncSetAttribute(prefill_state_kernel<K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                : cudaFuncSetAttribute(prefill_fused_kernel<K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[two][dev] = context_key();
    }
    int *status = device_status_ptr();
    const CUtensorMap &mxo = mx ? *mx : mo;  // the X map (unused unless kFirstX)
    auto launch = [&](long long grid, SegPlan plan) {
        if (two && plan.mode != kSecond && K == 64)
            // right after the key-side pass: its tail overlaps this grid's
            // prologue (the issuer waits for it before the first load).
            // Measured on the 8 x 4096 x 16 prefill: d_k' = 64 gains 6 us
            // (0.220 -> 0.214 ms); at d_k = 128 the state CTAs, placed on
            // whichever SMs the key-side pass frees first, ran 10 us slower,
            // so that width keeps the plain launch
            return launch_pdl(prefill_state_kernel<K>, (unsigned)grid, kTcThreads, smem, stream,
                              mq, mk, mv, mo, mxo, alpha, beta, S0, o != nullptr, ST, T, Ts, H,
                              (int)BH, plan, prep, status);
        if (two)
            prefill_state_kernel<K><<<(unsigned)grid, kTcThreads, smem, stream>>>(
                mq, mk, mv, mo, mxo, alpha, beta, S0, o != nullptr, ST, T, Ts, H, (int)BH, plan,
                prep, status);
        else
            prefill_fused_kernel<K><<<(unsigned)grid, kFuThreads, smem, stream>>>(
                mq, mk, mv, mo, alpha, beta, S0, o != nullptr, ST, T, Ts, H, (int)BH, plan,
                status);
        return cudaGetLastError();
    };
    if (sh.nseg == 1) return launch(BH, SegPlan{kWhole, 1, T, nullptr});
    // no second pass: the two-pass form when it has the X buffer or no outputs
    const bool corr = two && (o == nullptr || (mx != nullptr && xbuf != nullptr));
    cudaError_t e = launch(BH * (2 * sh.nseg - 1),
                           SegPlan{corr && o ? kFirstX : kFirst, sh.nseg, sh.seg_len, ws});
    if (e != cudaSuccess) return e;
    static uintptr_t comb_set[64] = {};
    if (comb_set[dev] != context_key()) {
        e = cudaFuncSetAttribute(segment_combine_kernel<K>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)CombineLayout<K>::SMEM);
        if (e != cudaSuccess) return e;
        comb_set[dev] = context_key();
    }
    segment_combine_kernel<K><<<dim3((unsigned)BH, 128 / 16), 256, CombineLayout<K>::SMEM,
                                stream>>>(ws, (int)BH, sh.nseg, corr ? ST : nullptr);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!corr) return launch(BH * (sh.nseg - 1), SegPlan{kSecond, sh.nseg, sh.seg_len, ws});
    if (o == nullptr) return cudaSuccess;
    using CL = CorrLayout<K>;
    static uintptr_t corr_set[64] = {};
    if (corr_set[dev] != context_key()) {
        e = cudaFuncSetAttribute(segment_correct_kernel<K>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CL::SMEM);
        if (e != cudaSuccess) return e;
        corr_set[dev] = context_key();
    }
    // splits of each segment's tiles: the grid within one wave of two CTAs per SM
    const long long cells = BH * (sh.nseg - 1);
    const int tiles = (sh.seg_len + 63) / 64;
    const int split = (int)std::max<long long>(
        1, std::min<long long>(tiles, 2LL * sm_count() / cells));
    if (BH > 0x7fffffffLL || sh.nseg - 1 > 65535) return cudaErrorInvalidConfiguration;
    segment_correct_kernel<K><<<dim3((unsigned)BH, (unsigned)(sh.nseg - 1), (unsigned)split),
                                kCorrThreads, CL::SMEM, stream>>>(
        ws, xbuf, static_cast<__nv_bfloat16 *>(o), T, Ts, H, (int)BH, sh.nseg, sh.seg_len, status);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_tc_t(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *ST, int B, int T,
                        int Ts, int H, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_token_map(&mq, q, B, T, Ts, H, K) || !make_token_map(&mk, k, B, T, Ts, H, K) ||
        !make_token_map(&mv, v, B, T, Ts, H, 128))
        return cudaErrorInvalidValue;
    // outputs go out by TMA store (the map is unused without outputs)
    if (o) {
        if (!make_token_map(&mo, o, B, T, Ts, H, 128)) return cudaErrorInvalidValue;
    } else {
        mo = mv;
    }
    const long long BH = (long long)B * H;
    const SegShape sh = segment_shape(B * H, T, K, sm_count());
    if (sh.nseg == 1 && BH > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (sh.nseg > 1) {
        if (!workspace || workspace_bytes < sh.workspace_bytes) return cudaErrorInvalidValue;
        if (BH * (2 * sh.nseg - 1) > 0x7fffffffLL || BH > 65535)
            return cudaErrorInvalidConfiguration;
    }
    float *ws = static_cast<float *>(workspace);
    // Two-pass form when the workspace also holds every chunk's key-side operands.
    const size_t prep_off = prefill_prep_offset(sh);
    const size_t need = prep_off + prefill_prep_bytes(BH, T);
    if (workspace && workspace_bytes >= need) {
        uint8_t *prep = static_cast<uint8_t *>(workspace) + prep_off;
        // segments' X buffer after the operands, when the workspace holds it
        const size_t xbytes = prefill_x_bytes(sh, BH, T);
        CUtensorMap mx;
        __nv_bfloat16 *xbuf = nullptr;
        if (xbytes > 0 && workspace_bytes >= need + xbytes) {
            xbuf = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(workspace) + need);
            if (!make_token_map(&mx, xbuf, B, T, T, H, 128)) return cudaErrorInvalidValue;
        }
        const cudaError_t e = launch_prep<K>(mq, mk, alpha, beta, prep, BH, T, Ts, H, stream);
        if (e != cudaSuccess) return e;
        return run_tc<K>(mq, mk, mv, mo, alpha, beta, S0, o, ST, BH, T, Ts, H, sh, ws, prep,
                         stream, xbuf ? &mx : nullptr, xbuf);
    }
    return run_tc<K>(mq, mk, mv, mo, alpha, beta, S0, o, ST, BH, T, Ts, H, sh, ws, nullptr,
                     stream);
}

}  // namespace

// Number of segments for B*H sequences of T tokens on `nsm` SMs: a cost model
// in chunk-times.  One CTA per sequence costs ceil(BH / nsm) waves of the
// whole length; with P segments the first pass runs BH (2P - 1) CTAs and the
// second BH (P - 1), each over T / P tokens, plus the combine (~0.6 chunk-time
// per segment) and a ~2 chunk-time start-up per wave.
SegShape segment_shape(int BH, int T, int K, int nsm) {
    SegShape sh{1, T, 0};
    const int nchunks = (T + 63) / 64;
    if (nsm < 2 || BH < 1 || BH * 2 > nsm || nchunks < 16) return sh;
    auto waves = [&](long long ctas) { return (double)((ctas + nsm - 1) / nsm); };
    double best = (nchunks + 2) * waves(BH);
    int bestP = 1;
    for (int P = 2; P <= 64 && nchunks / P >= 4; ++P) {
        const int segc = (nchunks + P - 1) / P;
        const double cost = (segc + 2) * (waves((long long)BH * (2 * P - 1)) +
                                          waves((long long)BH * (P - 1))) + 0.6 * P;
        if (cost < best) { best = cost; bestP = P; }
    }
    if (bestP == 1) return sh;
    const int segc = (nchunks + bestP - 1) / bestP;
    sh.seg_len = segc * 64;
    sh.nseg = (T + sh.seg_len - 1) / sh.seg_len;
    if (sh.nseg < 2) return SegShape{1, T, 0};
    sh.workspace_bytes = 3ull * BH * sh.nseg * 128ull * K * sizeof(float);
    return sh;
}

size_t prefill_prep_offset(const SegShape &sh) {
    return sh.nseg > 1 ? (sh.workspace_bytes + 255) & ~size_t(255) : 0;
}
size_t prefill_x_bytes(const SegShape &sh, long long BH, int T) {
    return sh.nseg > 1 ? ((size_t)BH * (size_t)T * 128 * sizeof(__nv_bfloat16) + 255) & ~size_t(255)
                       : 0;
}
size_t prefill_prep_bytes(long long BH, int T) {
    return (size_t)BH * (size_t)((T + 63) / 64) * kPrepChunkBytes;
}

// Workspace of the gathering prefill: segment slots, every chunk's key-side
// operands, then the gathered q' and k' ([B, T, H, 64] bf16 each).
GatheredLayout gathered_layout(int B, int T, int H) {
    GatheredLayout g{};
    const SegShape sh = segment_shape(B * H, T, 64, sm_count());
    g.prep = prefill_prep_offset(sh);
    const size_t tok = (size_t)B * T * H * 64 * sizeof(__nv_bfloat16);
    g.qg = (g.prep + prefill_prep_bytes((long long)B * H, T) + 255) & ~size_t(255);
    g.kg = (g.qg + tok + 255) & ~size_t(255);
    g.x = (g.kg + tok + 255) & ~size_t(255);
    g.total = g.x + prefill_x_bytes(sh, (long long)B * H, T);
    return g;
}

cudaError_t launch_prefill_gathered(const void *q_full, const void *k_full, const int *idx,
                                    const void *v, const float *alpha, const float *beta,
                                    const float *S0, void *o, float *ST, int B, int T, int H,
                                    void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const GatheredLayout g = gathered_layout(B, T, H);
    if (!workspace || workspace_bytes < g.total) return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto *qg = reinterpret_cast<__nv_bfloat16 *>(ws + g.qg);
    auto *kg = reinterpret_cast<__nv_bfloat16 *>(ws + g.kg);
    CUtensorMap mqf, mkf, mq, mk, mv, mo;
    if (!make_token_map(&mqf, q_full, B, T, T, H, 128) ||
        !make_token_map(&mkf, k_full, B, T, T, H, 128) || !make_token_map(&mq, qg, B, T, T, H, 64) ||
        !make_token_map(&mk, kg, B, T, T, H, 64) || !make_token_map(&mv, v, B, T, T, H, 128))
        return cudaErrorInvalidValue;
    if (o) {
        if (!make_token_map(&mo, o, B, T, T, H, 128)) return cudaErrorInvalidValue;
    } else {
        mo = mv;
    }
    const long long BH = (long long)B * H;
    const SegShape sh = segment_shape(B * H, T, 64, sm_count());
    if (BH * (2 * sh.nseg - 1) > 0x7fffffffLL || (sh.nseg > 1 && BH > 65535))
        return cudaErrorInvalidConfiguration;
    uint8_t *prep = ws + g.prep;
    // segments: the X buffer, as in the plain two-pass form
    CUtensorMap mx;
    __nv_bfloat16 *xbuf = nullptr;
    if (g.total > g.x) {
        xbuf = reinterpret_cast<__nv_bfloat16 *>(ws + g.x);
        if (!make_token_map(&mx, xbuf, B, T, T, H, 128)) return cudaErrorInvalidValue;
    }
    cudaError_t e = launch_prep<64, true>(mqf, mkf, alpha, beta, prep, BH, T, T, H, stream,
                                          PrepGather{idx, qg, kg});
    if (e != cudaSuccess) return e;
    return run_tc<64>(mq, mk, mv, mo, alpha, beta, S0, o, ST, BH, T, T, H, sh,
                      reinterpret_cast<float *>(ws), prep, stream, xbuf ? &mx : nullptr, xbuf);
}

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *ST, int B,
                              int T, int Ts, int H, int K, int V, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    if (V != 128) return cudaErrorInvalidValue;
    if (K == 128)
        return launch_tc_t<128>(q, k, v, alpha, beta, S0, o, ST, B, T, Ts, H, workspace,
                                workspace_bytes, stream);
    if (K == 64)
        return launch_tc_t<64>(q, k, v, alpha, beta, S0, o, ST, B, T, Ts, H, workspace,
                               workspace_bytes, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
