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
