"""Float64 numpy statement of the chunkwise form of the gated delta rule.

A design aid for the GPU prefill, not the oracle: the tests show it equals the
token-by-token oracle to rounding before any kernel relies on the algebra.

For one sequence and a chunk of C tokens with local cumulative log-decay
G_t = sum_{s<=t} log alpha_s (gamma_t = exp G_t, Gamma_ts = exp(G_t - G_s)):

  A_ts = beta_t Gamma_ts (k_t . k_s)  for s < t        (strictly lower)
  T    = (I + A)^{-1}                                   (unit lower)
  W    = T diag(beta gamma) K,   U~ = T diag(beta) V
  U    = U~ - W S0^T             rows are the pseudo-values u_t
  O    = diag(gamma) Q S0^T + (mask_{s<=t} Gamma_ts (q_t . k_s)) U
  S_C  = gamma_C S0 + U^T diag(exp(G_C - G_s)) K

derived by unrolling S_t = alpha_t S_{t-1} + u_t k_t^T with
u_t = beta_t (v_t - alpha_t S_{t-1} k_t) ("On State Reduction in Linear
Attention" notes, Sec. 2.3: the delta rule as an outer-product accumulation
of pseudo-values).  A ragged last chunk is padded with k = q = v = 0,
beta = 0, alpha = 1, which leaves every valid row unchanged.
"""
import numpy as np


def chunk_recurrence(q, k, v, alpha, beta, S0=None, C=64):
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    ST = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for c0 in range(0, T, C):
                n = min(C, T - c0)
                Kc = np.zeros((C, K)); Qc = np.zeros((C, K)); Vc = np.zeros((C, V))
                g = np.zeros(C); be = np.zeros(C)
                Kc[:n] = k[b, c0:c0 + n, h]; Qc[:n] = q[b, c0:c0 + n, h]
                Vc[:n] = v[b, c0:c0 + n, h]
                g[:n] = np.log(alpha[b, c0:c0 + n, h]); be[:n] = beta[b, c0:c0 + n, h]
                G = np.cumsum(g)
                gam = np.exp(G)
                Gam = np.exp(G[:, None] - G[None, :])
                lower = np.tril(np.ones((C, C)), -1)
                A = be[:, None] * Gam * (Kc @ Kc.T) * lower
                Tm = np.linalg.inv(np.eye(C) + A)
                W = Tm @ ((be * gam)[:, None] * Kc)
                Ut = Tm @ (be[:, None] * Vc)
                U = Ut - W @ S.T
                P = np.tril(Gam * (Qc @ Kc.T))
                O = gam[:, None] * (Qc @ S.T) + P @ U
                S = gam[-1] * S + U.T @ (np.exp(G[-1] - G)[:, None] * Kc)
                o[b, c0:c0 + n, h] = O[:n]
            ST[b, h] = S
    return o, ST


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 (ties to even), returned
    as float64: the rounding the kernels apply to their MMA operands."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def f32_round(x):
    """Round float64 values to float32 (returned as float64)."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def bf16_split(x, parts):
    """x as the sum of `parts` bfloat16 numbers: hi = bf16(x), then each
    next part the bf16 of what the float32 value still lacks."""
    out, rest = [], f32_round(x)
    for _ in range(parts):
        p = bf16_round(rest)
        out.append(p)
        rest = f32_round(rest - p)
    return out


def mm_bf16_split(a, b, parts):
    """a @ b on bf16 tensor cores with float32 operands split into `parts`
    bf16 parts: the products of part i of a and part j of b with i + j <
    parts (2 parts: hi hi + hi lo + lo hi), accumulated in float32."""
    A, Bp = bf16_split(a, parts), bf16_split(b, parts)
    acc = np.zeros((np.shape(a)[0], np.shape(b)[1]), np.float32)
    for i, ai in enumerate(A):
        for j, bj in enumerate(Bp):
            if i + j < parts:
                acc += ai.astype(np.float32) @ bj.astype(np.float32)
    return acc.astype(np.float64)


def _chunk_operands(k, q, v, alpha, beta, b, h, c0, C):
    """Zero-padded chunk tiles and its scalar-gate quantities."""
    T = k.shape[1]
    n = min(C, T - c0)
    K, V = k.shape[-1], v.shape[-1]
    Kc = np.zeros((C, K)); Qc = np.zeros((C, K)); Vc = np.zeros((C, V))
    g = np.zeros(C); be = np.zeros(C)
    Kc[:n] = k[b, c0:c0 + n, h]; Qc[:n] = q[b, c0:c0 + n, h]; Vc[:n] = v[b, c0:c0 + n, h]
    g[:n] = np.log(alpha[b, c0:c0 + n, h]); be[:n] = beta[b, c0:c0 + n, h]
    G = np.cumsum(g)
    gam = np.exp(G)
    Gam = np.exp(G[:, None] - G[None, :])
    A = be[:, None] * Gam * (Kc @ Kc.T) * np.tril(np.ones((C, C)), -1)
    Tm = np.linalg.inv(np.eye(C) + A)
    return dict(n=n, K=Kc, Q=Qc, V=Vc, beta=be, gam=gam, gC=gam[-1],
                dec=np.exp(G[-1] - G), P=np.tril(Gam * (Qc @ Kc.T)),
                Tp=Tm * (be * gam)[None, :], Tpp=Tm * be[None, :])


def chunk_state_chain(q, k, v, alpha, beta, S0=None, C=64, lookahead=False, rnd=None,
                      prod=None):
    """The state pass of the two-pass prefill, one sequence per (b, h), on the
    key-side operands T' = T diag(beta gamma), T'' = T diag(beta) and P.

    lookahead=False is the chain the kernel runs today (all quantities
    transposed as in the kernel: value channels on the rows):

      U^T(n) = U~^T(n) + S(n-1) NW(n),   NW = -W^T = -K^T T'^T,  U~^T = V^T T''^T
      O^T(n) = S(n-1) (gamma Q)^T + U^T(n) P^T
      S(n)   = gamma_n S(n-1) + U^T(n) diag(dec) K(n)

    lookahead=True forms U(n+1) without waiting for S(n): since
    S(n) NW(n+1) = S(n-1) [gamma_n NW(n+1)] + U^T(n) M(n) with
    M(n) = diag(dec_n) K(n) NW(n+1),

      U^T(n+1) = U~^T(n+1) + S(n-1) [gamma_n NW(n+1)] + U^T(n) M(n),

    the same U exactly (S(n) is still formed for O and the final state).
    rnd (e.g. bf16_round) is applied where the kernel rounds an MMA operand:
    T', T'', P, NW (and gamma_n NW, M), the state copy, U^T, U^T diag(dec)
    and gamma Q; products then accumulate in float32 and the state stays
    float32, as on the GPU.  prod, if given, forms every product instead
    (e.g. mm_bf16_split with rnd=f32_round: float32 operands on bf16 tensor
    cores).  Returns (o, S_T) like chunk_recurrence.
    """
    r = rnd if rnd is not None else (lambda x: x)
    acc = np.float32 if rnd is not None else np.float64
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    ST = np.zeros((B, H, V, K))
    mm = prod if prod is not None else (
        lambda a, b_: (np.asarray(a, acc) @ np.asarray(b_, acc)).astype(np.float64))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            S = S.astype(acc).astype(np.float64)
            ops = [_chunk_operands(k, q, v, alpha, beta, b, h, c0, C) for c0 in range(0, T, C)]
            nw = [r(-mm(c["K"].T, r(c["Tp"]).T)) for c in ops]     # -W^T(n), K x C
            ut = [mm(c["V"].T, r(c["Tpp"]).T) for c in ops]          # U~^T(n), V x C
            U_next = None
            for n, c in enumerate(ops):
                if not lookahead or n == 0:
                    Un = ut[n] + mm(r(S), nw[n])
                else:
                    Un = U_next
                Ub = r(Un)
                Ud = r(Un * c["dec"][None, :])
                if lookahead and n + 1 < len(ops):
                    M = r(c["dec"][:, None] * mm(c["K"], nw[n + 1]))  # rows scaled after
                    U_next = ut[n + 1] + mm(r(S), r(c["gC"] * nw[n + 1])) + mm(Ub, M)
                Ot = mm(r(S), r(c["gam"][:, None] * c["Q"]).T) + mm(Ub, r(c["P"]).T)
                S = (acc(c["gC"]) * S.astype(acc) + mm(Ud, c["K"]).astype(acc)).astype(np.float64)
                o[b, n * C:n * C + c["n"], h] = Ot.T[:c["n"]]
            ST[b, h] = S
    return o, ST


def kda_chunk_recurrence(q, k, v, alpha, beta, S0=None, C=64, sub=16, rnd=None):
    """Chunkwise form of KDA (per-key-channel decay alpha_t in R^K on the right
    of the state, scalar beta), with the per-channel exponents inside the
    intra-chunk products referred to the midpoint of each `sub`-token row
    block.  With G_t in R^K the in-chunk cumulative log-decay:

      A'_ts = beta_t sum_j k_tj k_sj e^(G_tj - G_sj)   (s < t)
      P'_ts = sum_j q_tj k_sj e^(G_tj - G_sj)         (s <= t)
      T = (I + A')^{-1},  W = T diag(beta) (K (.) e^G),  U~ = T diag(beta) V
      U = U~ - W S^T,     O = (Q (.) e^G) S^T + P' U
      S <- S diag(e^(G_C)) + U^T (K (.) e^(G_C - G))

    For row block I with reference token m (its midpoint), e^(G_t - G_s) =
    e^(G_t - G_m) e^(G_m - G_s): rows of block I use the left factor, columns
    s <= the block's last token the right one, so each block row of A' and P'
    is one product of two scaled operands, and every factor is at most
    e^(sub/2 max |log alpha|) (at most 1 for s before the block).  Returns
    (o, S_T, max_factor), max_factor the largest exponential formed.
    rnd (e.g. bf16_round) rounds every tensor-core operand as a kernel would
    (the scaled block operands, T diag(beta), the scaled keys and queries,
    the state copy, U, P'); products then accumulate in float32, the inverse
    and the state stay float32.
    """
    r = rnd if rnd is not None else (lambda x: x)
    acc = np.float32 if rnd is not None else np.float64
    mm = lambda a, b_: (np.asarray(a, acc) @ np.asarray(b_, acc)).astype(np.float64)
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    ST = np.zeros((B, H, V, K))
    fmax = 0.0
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for c0 in range(0, T, C):
                n = min(C, T - c0)
                Kc = np.zeros((C, K)); Qc = np.zeros((C, K)); Vc = np.zeros((C, V))
                lg = np.zeros((C, K)); be = np.zeros(C)
                Kc[:n] = k[b, c0:c0 + n, h]; Qc[:n] = q[b, c0:c0 + n, h]
                Vc[:n] = v[b, c0:c0 + n, h]
                lg[:n] = np.log(alpha[b, c0:c0 + n, h]); be[:n] = beta[b, c0:c0 + n, h]
                G = np.cumsum(lg, axis=0)                      # C x K
                A = np.zeros((C, C)); P = np.zeros((C, C))
                for i0 in range(0, C, sub):
                    m = i0 + sub // 2 - 1                      # the block's reference token
                    last = i0 + sub                            # columns s < last
                    lf = np.exp(G[i0:last] - G[m])             # rows t of block I
                    rf = np.exp(G[m] - G[:last])               # columns s <= last token
                    fmax = max(fmax, lf.max(), rf.max())
                    kt = r(Kc[i0:last] * lf)
                    qt = r(Qc[i0:last] * lf)
                    ks = r(Kc[:last] * rf)
                    A[i0:last, :last] = mm(kt, ks.T)
                    P[i0:last, :last] = mm(qt, ks.T)
                tt = np.arange(C)
                A = be[:, None] * A * (tt[None, :] < tt[:, None])
                P = P * (tt[None, :] <= tt[:, None])
                Tm = np.linalg.inv((np.eye(C) + A).astype(acc)).astype(np.float64)
                Tb = r(Tm * be[None, :])                        # T diag(beta)
                W = r(mm(Tb, r(Kc * np.exp(G))))
                Ut = mm(Tb, Vc)
                U = Ut - mm(W, r(S).T)
                Ub = r(U)
                O = mm(r(Qc * np.exp(G)), r(S).T) + mm(r(P), Ub)
                S = (S * np.exp(G[-1])[None, :]).astype(acc).astype(np.float64) + \
                    mm(Ub.T, r(Kc * np.exp(G[-1] - G)))
                o[b, c0:c0 + n, h] = O[:n]
            ST[b, h] = S
    return o, ST, fmax


def gdn2_chunk_recurrence(q, k, v, alpha, b_gate, w_gate, S0=None, C=64, sub=16):
    """Chunkwise form of GDN2: the KDA decay with a key-side erase gate b
    (erase direction e_t = b_t (.) k_t) and a value-side write gate w
    (content z_t = w_t (.) v_t); the outer products keep k_t on their right.
    KDA's algebra with beta_t k_t -> e_t in the rows of A and in W, and
    beta_t v_t -> z_t:

      A''_ts = sum_j e_tj k_sj e^(G_tj - G_sj)  (s < t),  T = (I + A'')^{-1}
      U = T Z - T (E (.) e^G) S^T,   O and S as for KDA,

    the exponents referred to each row block's midpoint as in
    kda_chunk_recurrence.  Float64; returns (o, S_T)."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    ST = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for c0 in range(0, T, C):
                n = min(C, T - c0)
                Kc = np.zeros((C, K)); Qc = np.zeros((C, K)); Ec = np.zeros((C, K))
                Zc = np.zeros((C, V)); lg = np.zeros((C, K))
                Kc[:n] = k[b, c0:c0 + n, h]; Qc[:n] = q[b, c0:c0 + n, h]
                Ec[:n] = b_gate[b, c0:c0 + n, h] * k[b, c0:c0 + n, h]
                Zc[:n] = w_gate[b, c0:c0 + n, h] * v[b, c0:c0 + n, h]
                lg[:n] = np.log(alpha[b, c0:c0 + n, h])
                G = np.cumsum(lg, axis=0)
                A = np.zeros((C, C)); P = np.zeros((C, C))
                for i0 in range(0, C, sub):
                    m = i0 + sub // 2 - 1
                    last = i0 + sub
                    lf = np.exp(G[i0:last] - G[m])
                    ks = Kc[:last] * np.exp(G[m] - G[:last])
                    A[i0:last, :last] = (Ec[i0:last] * lf) @ ks.T
                    P[i0:last, :last] = (Qc[i0:last] * lf) @ ks.T
                tt = np.arange(C)
                A = A * (tt[None, :] < tt[:, None])
                P = P * (tt[None, :] <= tt[:, None])
                Tm = np.linalg.inv(np.eye(C) + A)
                U = Tm @ Zc - (Tm @ (Ec * np.exp(G))) @ S.T
                O = (Qc * np.exp(G)) @ S.T + P @ U
                S = S * np.exp(G[-1])[None, :] + U.T @ (Kc * np.exp(G[-1] - G))
                o[b, c0:c0 + n, h] = O[:n]
            ST[b, h] = S
    return o, ST
