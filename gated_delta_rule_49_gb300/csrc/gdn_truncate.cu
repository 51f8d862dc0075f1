// Rank-r truncation of states ("How much of a Gated DeltaNet state is used"
// blog, Sec. 3): S <- U_r U_r^T S, U_r the left singular vectors of the r
// largest singular values, plus the singular values themselves.
//
// One CTA per state.  First a Householder QR, S = Q R (Q is not formed; the
// columns in registers, 16 per warp, one barrier per reflector): the Jacobi
// sweeps then run on the K columns of R^T, which are much closer to
// orthogonal than those of S (the preconditioned one-sided Jacobi SVD; on
// the prefill's final states the slowest state needs 9 to 10 sweeps instead
// of 19 to 20).  With
// R^T J = U_x Sigma the columns of U_x are the right singular vectors of S,
// so Y = S U_x = (Q J) Sigma has column norms sigma_c (formed against the
// original S), and S_r = Y_r U_x,r^T.
// One-sided (Hestenes) Jacobi on the K columns of R^T, with the columns held
// in registers in blocks of four: a group of 16 lanes (half a warp) holds a
// pair of blocks, K / 16 entries of each of its 8 columns per lane (runs of
// four: lane l holds entries 64 i + 4 l .. + 3), so a state takes K / 8
// groups (8 warps for K = 128, two per scheduler).  A sweep visits every
// column pair once:
//   - block rounds: each group rotates the 16 cross pairs of its two blocks,
//     in four mini-rounds of four disjoint pairs (top column i with bottom
//     column (i + m) % 4); then the blocks move to the next arrangement of
//     the round-robin (circle method: block 0 stays, the others step around a
//     cycle) through shared memory, as 16-byte runs.  K/4 - 1 block rounds
//     meet every pair of blocks once and return them to their places.
//   - in the first block round also the 6 pairs inside each block: three
//     rounds of the fixed pairs (0,3) (1,2) of each block, its columns 1..3
//     stepping around between rounds (the circle method again).
// Each mini-round sums its four dot products with a reduce-scatter over the
// 16 lanes, so lane quad k (lanes 4k .. 4k + 3) ends with pair k's sum and
// computes that pair's rotation once; the quads then broadcast (c, s).  The
// quad also carries its pair's two squared norms.  (Measured on the 128
// final states of the 8 x 4096 x 16 prefill: blocks of four in 8 warps per
// state beat blocks of eight in 4 warps, whose one warp per scheduler leaves
// the rotations' latencies exposed, and blocks of two in 16 warps, whose
// shorter blocks spend more instructions per pair.)
// The rotation makes the pair orthogonal:
//
//   a = |c_p|^2, b = |c_q|^2, g = c_p . c_q,  zeta = (b - a) / (2 g),
//   t = sign(zeta) / (|zeta| + sqrt(1 + zeta^2)),  c = 1/sqrt(1 + t^2), s = c t,
//   c_p <- c c_p - s c_q,   c_q <- s c_p + c c_q,   a <- a - t g,  b <- b + t g
//
// (a and b are recomputed from the columns at every block round; within one
// the updates above carry them).  It is skipped when |g| <= sqrt(V) eps
// sqrt(a b) (columns orthogonal to float32 precision) or |g| <= 1e-12 |S|_F^2
// (a coupling far below anything that can move the singular values or
// subspaces at float32 precision; without this floor the noise-level columns
// of a low-rank state keep the sweeps going).  The rotation uses fast
// reciprocal / square-root forms: an angle that is off in the last bits
// leaves a residual the next sweep removes.  Sweeps repeat until one rotates
// nothing (or max_sweeps; then the not-converged status bit is set).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kLanes = 16;  // lanes of one column (half a warp)
constexpr int kBlk = 4;     // columns per block
// Orthogonality threshold |g| <= sqrt(n) eps sqrt(a b) for columns of length
// n, eps = 2^-24 (float32).
template <int N>
__host__ __device__ constexpr float jacobi_tol() {
    return N == 128 ? 6.75e-7f : N == 64 ? 4.77e-7f : 3.38e-7f;
}

template <int V, int K>
struct TruncLayout {
    static constexpr int E = K / kLanes;    // entries of a column of R^T per lane
    static constexpr int NB = K / kBlk;     // blocks
    static constexpr int NS = NB / 2;       // block pairs = lane groups (8 columns each)
    static constexpr int NT = NS * kLanes;  // threads (16 columns per warp in the QR)
    static constexpr int LDT = K + 4;       // row stride of U_x [K][LDT]
    // columns of a thread's 8-row output tile (at least one float4): TK of
    // S_r [V][K], TV of Y^T [K][V]
    static constexpr int TK = K * K / (NT * 8) > 4 ? K * K / (NT * 8) : 4;
    static constexpr int TV = K * V / (NT * 8) > 4 ? K * V / (NT * 8) : 4;
    // shared memory, in floats
    static constexpr int BOARD0 = 0;                // QR reflectors; board [K][K]; U_x [K][LDT]
    static constexpr int BOARD1 = BOARD0 + K * LDT; // board [K][K]; U_x^T [K][K] at the end
    static constexpr int SC = BOARD1 + K * K;       // [V][K] the original S; Y^T [K][V]
    static constexpr int NRM = SC + V * K;          // [K] diag(R), then 1 / column norms
    static constexpr int SIG = NRM + K;             // [K] sigma^2
    static constexpr int SEL = SIG + K;             // [K] column of rank i (int)
    static constexpr size_t BYTES = (size_t)(SEL + K) * 4;
    static_assert(V % kLanes == 0 && K % (2 * kBlk) == 0 && K <= V && NT == 2 * K, "shape");
    static_assert(TK % 4 == 0 && K % TK == 0 && TV % 4 == 0 && V % TV == 0, "tiles");
    static_assert((K / 8) * (V / TV) <= NT, "one Y^T tile per thread at most");
};

// Sum four per-lane values over the 16 lanes of the group, scattering: lane
// quad k (lanes 4k .. 4k + 3, k = lane bits 3 and 2) gets the sum of x[k].
// The quad's four lanes hold the same sum (the last two levels add the same
// pairs, in either order).
__device__ __forceinline__ float reduce_scatter4(const float (&x)[4], int l) {
    const bool b3 = l & 8, b2 = l & 4;
    float h[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? x[i] : x[i + 2], keep = b3 ? x[i + 2] : x[i];
        h[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? h[0] : h[1], keep = b2 ? h[1] : h[0];
    float r = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

// The rotation of one pair from a = |c_p|^2, b = |c_q|^2, g = c_p . c_q:
// (c, s, t), or (1, 0, 0) when the pair is already orthogonal.  With
// d = b - a, h = 2 g, r = sqrt(d^2 + h^2) and u = |d| + r, the angle above
// (zeta = d / h) is t = sign(d) h / u, and 1 + t^2 = 2 r / u, so
//   c = u / sqrt(2 r u),  s = sign(d) h / sqrt(2 r u),  t = sign(d) h 2 r / (2 r u):
// two reciprocal square roots in sequence (each ~40 cycles) where the
// zeta form takes four.  The columns are scaled so that |S|_F ~ 1, which
// keeps d^2 + h^2 in range.
__device__ __forceinline__ bool jacobi_angle(float a, float b, float g, float floor_g, float tol2,
                                             float &c, float &s, float &t) {
    const bool rot = fabsf(g) > floor_g && g * g > tol2 * a * b;
    const float d = b - a, h = 2.f * g;
    const float x = fmaf(d, d, h * h);
    const float r = x * rsqrtf(x);
    const float u = fabsf(d) + r;
    const float rq = rsqrtf(2.f * r * u);
    const float sh = d >= 0.f ? h : -h;  // sign(d) h, sign(0) = +1
    c = rot ? u * rq : 1.f;
    s = rot ? sh * rq : 0.f;
    t = rot ? sh * (2.f * r) * (rq * rq) : 0.f;
    return rot;
}

// Rotate the four disjoint column pairs (P[k], Q[k]) of the group's registers,
// the quad of pair k computing its rotation: in cross mini-round M top k with
// bottom 4 + (k + M) % 4, or with INNER the pairs (0,3) (1,2) (4,7) (5,6)
// inside the blocks.  The quads of a warp may decide differently, so the
// rotation is predicated (c = 1, s = 0), and skipped as a whole when no pair
// of the warp rotates.  For the cross pairs the quad's squared norms (ap, aq)
// are given and updated (a <- a - t g, b <- b + t g); for the inner ones they
// are summed from the columns.
template <int E, bool INNER, int M = 0>
__device__ __forceinline__ void rotate4(float (&X)[8][E], int l, int gbase, float &ap, float &aq,
                                        float floor_g, float tol2, bool &any) {
    constexpr int P[4] = {0, 1, INNER ? 4 : 2, INNER ? 5 : 3};
    constexpr int Q[4] = {INNER ? 3 : 4 + M % 4, INNER ? 2 : 4 + (1 + M) % 4,
                          INNER ? 7 : 4 + (2 + M) % 4, INNER ? 6 : 4 + (3 + M) % 4};
    float gx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(X[P[k]][e], X[Q[k]][e], acc);
        gx[k] = acc;
    }
    const float g = reduce_scatter4(gx, l);
    if (INNER) {
        float ax[4], bx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float a0 = 0.f, b0 = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                a0 = fmaf(X[P[k]][e], X[P[k]][e], a0);
                b0 = fmaf(X[Q[k]][e], X[Q[k]][e], b0);
            }
            ax[k] = a0;
            bx[k] = b0;
        }
        ap = reduce_scatter4(ax, l);
        aq = reduce_scatter4(bx, l);
    }
    float c, s, t;
    const bool rot = jacobi_angle(ap, aq, g, floor_g, tol2, c, s, t);
    ap = fmaf(-t, g, ap);
    aq = fmaf(t, g, aq);
    if (__any_sync(0xffffffffu, rot)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float ck = __shfl_sync(0xffffffffu, c, gbase + 4 * k);
            const float sk = __shfl_sync(0xffffffffu, s, gbase + 4 * k);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = X[P[k]][e], y = X[Q[k]][e];
                X[P[k]][e] = fmaf(-sk, y, ck * x);
                X[Q[k]][e] = fmaf(sk, x, ck * y);
            }
        }
        any = true;
    }
}

// Between the cross mini-rounds quad k's next bottom column is the one quad
// k + 1 has just rotated: its norm comes from there.
__device__ __forceinline__ float next_bottom_norm(float aq, int l, int gbase) {
    return __shfl_sync(0xffffffffu, aq, gbase + ((l + 4) & 15));
}

// Columns 1..3 of each block step around (column j takes column j - 1,
// column 1 takes column 3; 3 steps cycle back).
template <int E>
__device__ __forceinline__ void step_inner(float (&X)[8][E]) {
#pragma unroll
    for (int b0 = 0; b0 < 8; b0 += 4)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float x = X[b0 + 3][e];
            X[b0 + 3][e] = X[b0 + 2][e];
            X[b0 + 2][e] = X[b0 + 1][e];
            X[b0 + 1][e] = x;
        }
}

// Squared norms of the quad's pair of columns (top k, bottom k).
template <int E>
__device__ __forceinline__ void quad_norms(const float (&X)[8][E], int l, float &ap, float &aq) {
    float ax[4], bx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float a0 = 0.f, b0 = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            a0 = fmaf(X[k][e], X[k][e], a0);
            b0 = fmaf(X[4 + k][e], X[4 + k][e], b0);
        }
        ax[k] = a0;
        bx[k] = b0;
    }
    ap = reduce_scatter4(ax, l);
    aq = reduce_scatter4(bx, l);
}

// Entry e of a column in lane l: runs of CH (4, or E when E < 4) entries,
// so a group's 16 lanes move a column as 16-byte (8-byte) pieces of one
// contiguous run.
template <int E>
__device__ __forceinline__ int entry_v(int e, int l) {
    constexpr int CH = E < 4 ? E : 4;
    return (e / CH) * (kLanes * CH) + l * CH + (e % CH);
}
template <int E, int V>
__device__ __forceinline__ void store_col(float *col, const float (&x)[E], int l) {
    if constexpr (E >= 4) {
#pragma unroll
        for (int i = 0; i < E / 4; ++i)
            *reinterpret_cast<float4 *>(col + entry_v<E>(4 * i, l)) =
                make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    } else {
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<float2 *>(col + entry_v<E>(e, l)) = make_float2(x[e], x[e + 1]);
    }
}
template <int E, int V>
__device__ __forceinline__ void load_col(const float *col, float (&x)[E], int l) {
    if constexpr (E >= 4) {
#pragma unroll
        for (int i = 0; i < E / 4; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(col + entry_v<E>(4 * i, l));
            x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const float2 v = *reinterpret_cast<const float2 *>(col + entry_v<E>(e, l));
            x[e] = v.x; x[e + 1] = v.y;
        }
    }
}
template <int V, int K>
__global__ void __launch_bounds__(TruncLayout<V, K>::NT, 1)
    truncate_kernel(float *__restrict__ Sg, int r, float *__restrict__ sigma, int max_sweeps,
                    int *status) {
    using L = TruncLayout<V, K>;
    constexpr int E = L::E, NS = L::NS, NT = L::NT, LDT = L::LDT, TK = L::TK, TV = L::TV;
    extern __shared__ __align__(16) float smf[];
    float *Sc = smf + L::SC;
    float *nrm = smf + L::NRM;
    float *sig2 = smf + L::SIG;
    int *sel = reinterpret_cast<int *>(smf + L::SEL);
    __shared__ float fro2;

    const int tid = threadIdx.x;
    const int grp = tid / kLanes, l = tid % kLanes;
    if (tid == 0) fro2 = 0.f;
    __syncthreads();
    float *Sh = Sg + (size_t)blockIdx.x * V * K;
    {
        // the original S
        float part = 0.f;
        for (int e4 = tid * 4; e4 < V * K; e4 += NT * 4) {
            const float4 x = *reinterpret_cast<const float4 *>(Sh + e4);
            part += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
            *reinterpret_cast<float4 *>(Sc + e4) = x;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if ((tid & 31) == 0) atomicAdd(&fro2, part);
    }

    // ---- Householder QR, S = Q R (Q is not formed) ----
    // Warp w owns columns w + NW cc (cc < 16, NW = K / 16 warps); its lane
    // group g (lanes 8 g .. 8 g + 7) holds cc = 4 g .. 4 g + 3, and lane slice
    // s = lane % 8 rows RP s .. RP s + RP - 1 of each (RP = V / 8), in
    // registers.  Step j reflects the columns right of j with
    // H_j = I - beta v v^T, v = A[j.., j] - alpha e_j, alpha = -sign(A[j][j]) |A[j.., j]|,
    // v_i = 0 above row j: v is published in shared memory (two buffers) by
    // the lane group owning column j, once its step j - 1 update of that
    // column is done; v^T a_c is a lane-local sum and a reduction over the
    // group's 8 lanes (the four columns of a group together).  Columns c <= j
    // take a zero step.  One barrier per step.  R[j][j] = alpha goes to nrm[j];
    // R[i][c], i < c, is row i of column c's registers when all is done.
    constexpr int NW = NT / 32, RP = V / 8;
    float *vbuf = smf + L::BOARD0;         // [2][V] reflectors (board 0 is free)
    float *bbuf = smf + L::BOARD0 + 2 * V; // [2] beta
    const int warp = tid >> 5, lane = tid & 31, qg = lane >> 3, qs = lane & 7;
    const unsigned gmask = 0xffu << (8 * qg);  // the lane group
    float a[4][RP];
    __syncthreads();  // the original S is in place
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < RP; ++k) a[q][k] = Sc[(RP * qs + k) * K + warp + NW * (4 * qg + q)];
    // the reflector of column c (this group's column q) from its rows >= c
    // after the earlier steps, into buffer c & 1 (called by the 8 lanes)
    auto publish = [&](const float (&x)[RP], int c) {
        float ss = 0.f, x0 = 0.f;
#pragma unroll
        for (int k = 0; k < RP; ++k) {
            const int row = RP * qs + k;
            if (row >= c) ss = fmaf(x[k], x[k], ss);
            if (row == c) x0 = x[k];
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(gmask, ss, off);
            x0 += __shfl_xor_sync(gmask, x0, off);  // one lane holds it, the rest 0
        }
        const float alpha = ss > 0.f ? -copysignf(sqrtf(ss), x0) : 0.f;
        const float den = ss - x0 * alpha;  // v^T v / 2 (>= ss)
        float *vb = vbuf + (c & 1) * V + RP * qs;
#pragma unroll
        for (int k = 0; k < RP; k += 4) {
            float o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int row = RP * qs + k + u;
                o[u] = row > c ? x[k + u] : row == c ? x0 - alpha : 0.f;
            }
            *reinterpret_cast<float4 *>(vb + k) = make_float4(o[0], o[1], o[2], o[3]);
        }
        if (qs == 0) {
            bbuf[c & 1] = den > 0.f ? 1.f / den : 0.f;
            nrm[c] = alpha;
        }
    };
    if (warp == 0 && qg == 0) publish(a[0], 0);
    for (int j = 0; j < K; ++j) {
        __syncthreads();  // reflector j published
        const float *vb = vbuf + (j & 1) * V + RP * qs;
        const float beta = bbuf[j & 1];
        float vv[RP];
#pragma unroll
        for (int k = 0; k < RP; k += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(vb + k);
            vv[k] = x.x; vv[k + 1] = x.y; vv[k + 2] = x.z; vv[k + 3] = x.w;
        }
        float d[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float e0 = 0.f, e1 = 0.f;
#pragma unroll
            for (int k = 0; k < RP; k += 2) {
                e0 = fmaf(vv[k], a[q][k], e0);
                e1 = fmaf(vv[k + 1], a[q][k + 1], e1);
            }
            d[q] = e0 + e1;
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[q] += __shfl_xor_sync(0xffffffffu, d[q], off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float t = warp + NW * (4 * qg + q) > j ? beta * d[q] : 0.f;
#pragma unroll
            for (int k = 0; k < RP; ++k) a[q][k] = fmaf(-t, vv[k], a[q][k]);
        }
        // the group owning column j + 1 publishes its reflector
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (warp + NW * (4 * qg + q) == j + 1) publish(a[q], j + 1);
    }
    // the columns of R^T (rows of R) into board 0, [K][K]: entry i of column
    // c is R[c][i], from row c of column i's registers
    __syncthreads();  // every read of the reflector buffers is done
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = warp + NW * (4 * qg + q);
#pragma unroll
        for (int k = 0; k < RP; ++k) {
            const int c = RP * qs + k;
            if (c < K) smf[L::BOARD0 + c * K + i] = c < i ? a[q][k] : c == i ? nrm[i] : 0.f;
        }
    }
    __syncthreads();

    // the sweeps run on the columns times 2^-e, |S|_F 2^-e in [0.5, 1): an
    // exact scaling (rotations do not depend on it) that keeps the angle's
    // squares in range (|R|_F = |S|_F); Y below is formed against the original S
    const int fe = fro2 > 0.f ? ilogbf(sqrtf(fro2)) + 1 : 0;
    const float scale = ldexpf(1.f, -fe);
    const float floor_g = 1e-12f * fro2 * scale * scale;
    const float tol2 = jacobi_tol<K>() * jacobi_tol<K>();

    // group grp holds columns 8 grp .. 8 grp + 7: its top block, then its bottom
    const int gbase = tid & 16;  // the group's first lane in its warp
    float X[8][E];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        load_col<E, K>(smf + L::BOARD0 + (8 * grp + j) * K, X[j], l);
#pragma unroll
        for (int e = 0; e < E; ++e) X[j][e] *= scale;
    }
    // where this group's blocks go at each move (board column of their first
    // column): the top steps to the next group's top (group 0's stays; the
    // last group's goes to its own bottom), the bottom to the previous
    // group's bottom (group 0's to group 1's top)
    const int top_to = grp == 0 ? 0 : grp == NS - 1 ? 8 * grp + 4 : 8 * (grp + 1);
    const int bot_to = grp == 0 ? 8 : 8 * (grp - 1) + 4;

    bool converged = false;
    for (int sweep = 0; sweep < max_sweeps && !converged; ++sweep) {
        bool any = false;
        for (int br = 0; br < L::NB - 1; ++br) {
            float ap, aq;  // squared norms of the quad's pair
            if (br == 0) {
#pragma unroll 1
                for (int rr = 0; rr < 3; ++rr) {
                    rotate4<E, true>(X, l, gbase, ap, aq, floor_g, tol2, any);
                    step_inner<E>(X);
                }
            }
            quad_norms<E>(X, l, ap, aq);
            rotate4<E, false, 0>(X, l, gbase, ap, aq, floor_g, tol2, any);
            aq = next_bottom_norm(aq, l, gbase);
            rotate4<E, false, 1>(X, l, gbase, ap, aq, floor_g, tol2, any);
            aq = next_bottom_norm(aq, l, gbase);
            rotate4<E, false, 2>(X, l, gbase, ap, aq, floor_g, tol2, any);
            aq = next_bottom_norm(aq, l, gbase);
            rotate4<E, false, 3>(X, l, gbase, ap, aq, floor_g, tol2, any);
            // move the blocks (boards alternate, so one barrier per round:
            // a board is rewritten only after the round that read it)
            float *bd = smf + ((br & 1) ? L::BOARD0 : L::BOARD1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                store_col<E, K>(bd + (top_to + j) * K, X[j], l);
                store_col<E, K>(bd + (bot_to + j) * K, X[4 + j], l);
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 8; ++j) load_col<E, K>(bd + (8 * grp + j) * K, X[j], l);
        }
        converged = __syncthreads_or(any) == 0;
    }
    if (!converged && tid == 0 && status) atomicOr(status, kStatusNotConverged);

    // U_x (the converged columns, unnormalised) into board 0 as [K][LDT], and
    // 1 / |c| per column.  Their lengths are not used as singular values:
    // rotations that are orthogonal only to rounding let the lengths drift
    // over a few thousand rotations while the directions stay accurate.  So
    // Y = S U_x is formed against the original S and sigma_c = |Y[:, c]|.
    float *Ux = smf + L::BOARD0;   // [K][LDT]: entry k of column c at [k][c]
    float *UxT = smf + L::BOARD1;  // [K][K]: column c contiguous
    float *Yt = Sc;                // [K][V], over the original S once it is read
    __syncthreads();  // every thread has read its last blocks from the boards
    {
        float ap, aq;
        quad_norms<E>(X, l, ap, aq);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < E; ++e) Ux[entry_v<E>(e, l) * LDT + 8 * grp + j] = X[j][e];
            store_col<E, K>(UxT + (8 * grp + j) * K, X[j], l);
        }
        if ((l & 3) == 0) {
            nrm[8 * grp + l / 4] = ap > 0.f ? rsqrtf(ap) : 0.f;
            nrm[8 * grp + 4 + l / 4] = aq > 0.f ? rsqrtf(aq) : 0.f;
        }
    }
    __syncthreads();
    // Y^T[c][v] = (1/|c|) sum_k U_x[k][c] S[v][k] against the original S:
    // one 8 x TV tile per thread, the lanes of a warp on consecutive column
    // tiles (so the rows of S they read are shared), k four at a time; the
    // tiles are written over S after every thread has read it
    const bool has_tile = tid < (K / 8) * (V / TV);
    const int c0 = (tid % (K / 8)) * 8, v0 = (tid / (K / 8)) * TV;
    float acc[8][TV];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TV; ++j) acc[i][j] = 0.f;
    if (has_tile) {
        for (int k = 0; k < K; k += 4) {
            float sv[TV][4];
#pragma unroll
            for (int j = 0; j < TV; ++j) {
                const float4 x = *reinterpret_cast<const float4 *>(Sc + (v0 + j) * K + k);
                sv[j][0] = x.x; sv[j][1] = x.y; sv[j][2] = x.z; sv[j][3] = x.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 a0 = *reinterpret_cast<const float4 *>(Ux + (k + u) * LDT + c0);
                const float4 a1 = *reinterpret_cast<const float4 *>(Ux + (k + u) * LDT + c0 + 4);
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < TV; ++j) acc[i][j] = fmaf(a[i], sv[j][u], acc[i][j]);
            }
        }
    }
    __syncthreads();
    if (has_tile) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float ni = nrm[c0 + i];
#pragma unroll
            for (int j = 0; j < TV; j += 4)
                *reinterpret_cast<float4 *>(Yt + (c0 + i) * V + v0 + j) =
                    make_float4(acc[i][j] * ni, acc[i][j + 1] * ni, acc[i][j + 2] * ni,
                                acc[i][j + 3] * ni);
        }
    }
    __syncthreads();
    for (int c = tid; c < K; c += NT) {
        float s2 = 0.f;
        for (int v = 0; v < V; ++v) s2 = fmaf(Yt[c * V + v], Yt[c * V + v], s2);
        sig2[c] = s2;
    }
    __syncthreads();
    for (int c = tid; c < K; c += NT) {  // rank of each column, ties by index
        const float sc = sig2[c];
        int rank = 0;
        for (int j = 0; j < K; ++j) rank += (sig2[j] > sc) || (sig2[j] == sc && j < c);
        sel[rank] = c;
    }
    __syncthreads();
    if (sigma)
        for (int i = tid; i < K; i += NT) sigma[(size_t)blockIdx.x * K + i] = sqrtf(sig2[sel[i]]);
    if (r >= K) return;  // nothing to cut (K <= V for every supported variant)

    // S <- Y_r U_x,r^T: 8 x TK tiles of [V][K]
    for (int tile = tid; tile < (V / 8) * (K / TK); tile += NT) {
        const int v0 = (tile / (K / TK)) * 8, k0 = (tile % (K / TK)) * TK;
        float acc[8][TK];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < TK; ++j) acc[i][j] = 0.f;
        for (int jr = 0; jr < r; ++jr) {
            const int c = sel[jr];
            const float nc = nrm[c];
            const float4 y0 = *reinterpret_cast<const float4 *>(Yt + c * V + v0);
            const float4 y1 = *reinterpret_cast<const float4 *>(Yt + c * V + v0 + 4);
            const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
            float u[TK];
#pragma unroll
            for (int j = 0; j < TK; j += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(UxT + c * K + k0 + j);
                u[j] = x.x * nc; u[j + 1] = x.y * nc; u[j + 2] = x.z * nc; u[j + 3] = x.w * nc;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < TK; ++j) acc[i][j] = fmaf(y[i], u[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < TK; j += 4)
                *reinterpret_cast<float4 *>(Sh + (size_t)(v0 + i) * K + k0 + j) =
                    make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
    }
}

template <int V, int K>
cudaError_t launch_trunc_t(float *S, int BH, int r, float *sigma, int max_sweeps,
                           cudaStream_t stream) {
    using L = TruncLayout<V, K>;
    auto kern = truncate_kernel<V, K>;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] != context_key()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    kern<<<BH, L::NT, L::BYTES, stream>>>(S, r, sigma, max_sweeps, device_status_ptr());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_truncate(float *S, int BH, int V, int K, int r, float *sigma,
                                  int max_sweeps, cudaStream_t stream) {
    if (V == 128 && K == 128) return launch_trunc_t<128, 128>(S, BH, r, sigma, max_sweeps, stream);
    if (V == 128 && K == 64) return launch_trunc_t<128, 64>(S, BH, r, sigma, max_sweeps, stream);
    if (V == 32 && K == 32) return launch_trunc_t<32, 32>(S, BH, r, sigma, max_sweeps, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
