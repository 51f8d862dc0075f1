"""Float64 CPU oracle for the gated delta-rule recurrence and its stable rank.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of what the GPU
path computes, written for a reader to check by eye.  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import it; the
product library never does, and the two share no code.

Functions
---------
recurrence(q, k, v, alpha, beta, S0=None, mode="gdn", threads=None)
    Token-by-token recurrence in float64 (C, ``gdn_oracle.c``).  Follows
    "On State Reduction in Linear Attention" notes, Sec. 2.1, Eqs. (1)-(2)
    (error-correction form of the delta rule, read o_t = S_t q_t, scalar decay
    of Gated DeltaNet) and "Linear Attention Architectures" notes, Sec. 2.4,
    Eqs. 15-17 (decay the old state first, then form the error).
stable_rank(S)
    ||S||_F^2, sigma_1 and er(S) = ||S||_F^2 / ||S||_2^2, the stable rank of
    "On State Reduction in Linear Attention" notes, Sec. 2.2, Eq. (5); sigma_1
    comes from LAPACK's SVD (numpy), a library routine independent of the GPU
    power iteration.  For S = 0 the ratio is undefined (the notes define it
    for nonzero states); this oracle returns (0, 0, 0) there.

recurrence_gated(q, k, v, alpha, beta=None, b=None, w=None, S0=None, gate="kda")
    The channel-gated rules of "Linear Attention Architectures" notes,
    Sec. 2.5 (KDA: per-key-channel decay on the right of the state, scalar
    beta) and Sec. 2.6 (GDN2: key-side erase gate b, value-side write gate
    w), token by token in float64 (C, ``gdn_oracle_gated.c``).
truncate_state(S, r)
    Rank-r truncation of "How much of a Gated DeltaNet state is used" blog,
    Sec. 3: project each state onto its top-r left singular directions,
    S_r = U_r U_r^T S (LAPACK SVD); r >= min(V, K) leaves S unchanged.
recurrence_truncated(q, k, v, alpha, beta, S0=None, seg_len=256, r=...)
    The same blog section's experiment: run the recurrence in segments of
    seg_len tokens and truncate the carried state to rank r at every segment
    boundary inside the sequence (the final state is not truncated).
channel_gram(k, q)
    G_h = K_h^T K_h + Q_h^T Q_h = M_h^T M_h for M_h = [K_cal; Q_cal] of head h
    ("On State Reduction in Linear Attention" notes, Sec. 2.8), float64.
drrqr(M, k, f=2.0, max_swaps=...)
    The same section's DRRQR channel selector: column-pivoted QR (LAPACK
    geqp3) for the initial permutation, then strong-RRQR swaps while the
    largest rho_ij = sqrt(U_ij^2 + (gamma_j / omega_i)^2) exceeds f, with
    U = A_k^{-1} B_k, omega_i = 1 / |row i of A_k^{-1}|, gamma_j = |column j of
    C_k|; returns the first k channels of the final permutation.
gather_normalize(x, idx, eps=1e-12)
    Channel selection with the normalisation recomputed on the kept
    coordinates ("On State Reduction in Linear Attention" notes, Sec. 2.6 and
    Alg. 1): y[..., h, :] = P_I x / max(|P_I x|, eps) with P_I the rows
    idx[h] of the identity.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, worked examples and invariants fixed by the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "gdn_oracle_gated.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODES = {"gdn": 0, "linear": 1}


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into ``liboracle.so`` with gcc (plain
    -O2, no architecture-specific flags, so it builds the same on x86 and Arm)."""
    stale = not os.path.exists(_LIB) or any(
        os.path.getmtime(_LIB) < os.path.getmtime(src) for src in _SRCS)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, *_SRCS, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.gdn_oracle_recurrence.argtypes = [dp] * 8 + [ctypes.c_int] * 7
            lib.gdn_oracle_recurrence.restype = ctypes.c_int
            lib.gdn_oracle_gated.argtypes = [dp] * 10 + [ctypes.c_int] * 7
            lib.gdn_oracle_gated.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, alpha, beta, S0=None, mode="gdn", threads=None, want_o=True):
    """Run the recurrence over every (batch, head) sequence.

    q, k: [B, T, H, K]; v: [B, T, H, V]; alpha, beta: [B, T, H];
    S0: [B, H, V, K] or None (zero state).  Inputs are upcast to float64 from
    whatever exact values the caller passes (bf16- or fp32-rounded).
    Returns (o [B, T, H, V] or None, S_T [B, H, V, K]) in float64.
    """
    k = _as_f64(k)
    B, T, H, K = k.shape
    v = _as_f64(v)
    V = v.shape[-1]
    q = _as_f64(q) if q is not None else None
    alpha = _as_f64(alpha)
    beta = _as_f64(beta)
    assert v.shape == (B, T, H, V)
    assert alpha.shape == (B, T, H) and beta.shape == (B, T, H)
    if q is not None:
        assert q.shape == (B, T, H, K)
    S0a = None
    if S0 is not None:
        S0a = _as_f64(S0)
        assert S0a.shape == (B, H, V, K)
    o = np.empty((B, T, H, V), dtype=np.float64) if (want_o and q is not None) else None
    ST = np.empty((B, H, V, K), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _load().gdn_oracle_recurrence(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0a), _ptr(o), _ptr(ST),
        B, T, H, K, V, MODES[mode], int(threads),
    )
    if rc != 0:
        raise RuntimeError(f"oracle recurrence failed with code {rc}")
    return o, ST


GATES = {"kda": 1, "gdn2": 2}


def recurrence_gated(q, k, v, alpha, beta=None, b=None, w=None, S0=None, gate="kda",
                     threads=None, want_o=True):
    """KDA (gate="kda": alpha [B,T,H,K], beta [B,T,H]) or GDN2 (gate="gdn2":
    alpha [B,T,H,K], b [B,T,H,K], w [B,T,H,V]).  Returns (o, S_T) in float64
    with the shapes of ``recurrence``."""
    k = _as_f64(k)
    B, T, H, K = k.shape
    v = _as_f64(v)
    V = v.shape[-1]
    q = _as_f64(q) if q is not None else None
    alpha = _as_f64(alpha)
    assert v.shape == (B, T, H, V) and alpha.shape == (B, T, H, K)
    betaa = ba = wa = None
    if gate == "kda":
        betaa = _as_f64(beta)
        assert betaa.shape == (B, T, H)
    else:
        ba, wa = _as_f64(b), _as_f64(w)
        assert ba.shape == (B, T, H, K) and wa.shape == (B, T, H, V)
    S0a = None
    if S0 is not None:
        S0a = _as_f64(S0)
        assert S0a.shape == (B, H, V, K)
    o = np.empty((B, T, H, V), dtype=np.float64) if (want_o and q is not None) else None
    ST = np.empty((B, H, V, K), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _load().gdn_oracle_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(betaa), _ptr(ba), _ptr(wa), _ptr(S0a),
        _ptr(o), _ptr(ST), B, T, H, K, V, GATES[gate], int(threads),
    )
    if rc != 0:
        raise RuntimeError(f"gated oracle failed with code {rc}")
    return o, ST


def stable_rank(S):
    """Return (fro2, sigma1, er) per matrix for S of shape [..., V, K].

    fro2 = sum of squared entries; sigma1 = largest singular value (LAPACK);
    er = fro2 / sigma1^2, and 0 where S is exactly zero.
    """
    S = _as_f64(S)
    lead = S.shape[:-2]
    M = S.reshape((-1,) + S.shape[-2:])
    fro2 = np.einsum("nij,nij->n", M, M)
    sig = np.linalg.svd(M, compute_uv=False)
    sigma1 = sig[:, 0] if sig.shape[1] else np.zeros(M.shape[0])
    er = np.zeros_like(fro2)
    nz = sigma1 > 0
    er[nz] = fro2[nz] / sigma1[nz] ** 2
    return fro2.reshape(lead), sigma1.reshape(lead), er.reshape(lead)


def truncate_state(S, r):
    """S [..., V, K] -> float64 U_r U_r^T S, U_r the left singular vectors of
    the r largest singular values of each state."""
    S = _as_f64(S)
    V, K = S.shape[-2:]
    if r >= min(V, K):
        return S.copy()
    U, _, _ = np.linalg.svd(S, full_matrices=False)
    Ur = U[..., :, :r]
    return Ur @ (np.swapaxes(Ur, -1, -2) @ S)


def recurrence_truncated(q, k, v, alpha, beta, S0=None, seg_len=256, r=None, threads=None):
    """Segments [0, L), [L, 2L), ...: run ``recurrence`` on each from the
    carried state, then replace that state by ``truncate_state(S, r)`` if the
    segment does not end the sequence.  Returns (o, S_T) in float64."""
    k = _as_f64(k)
    B, T, H, K = k.shape
    V = np.asarray(v).shape[-1]
    o = np.empty((B, T, H, V), dtype=np.float64)
    S = None if S0 is None else _as_f64(S0)
    if T == 0:
        return o, (np.zeros((B, H, V, K)) if S is None else S.copy())
    for t0 in range(0, T, seg_len):
        t1 = min(T, t0 + seg_len)
        sl = slice(t0, t1)
        o[:, sl], S = recurrence(np.asarray(q)[:, sl], k[:, sl], np.asarray(v)[:, sl],
                                 np.asarray(alpha)[:, sl], np.asarray(beta)[:, sl], S0=S,
                                 threads=threads)
        if t1 < T:
            S = truncate_state(S, r)
    return o, S


def channel_gram(k, q):
    """k, q [..., H, K] (any leading token axes) -> [H, K, K] float64."""
    k = _as_f64(k)
    q = _as_f64(q)
    H, K = k.shape[-2:]
    kf = k.reshape(-1, H, K)
    qf = q.reshape(-1, H, K)
    return np.einsum("nhi,nhj->hij", kf, kf) + np.einsum("nhi,nhj->hij", qf, qf)


def rrqr_factors(R, k):
    """From the upper-triangular R of M P (columns in the current order):
    A_k, B_k, C_k and the rho matrix of the strong-RRQR test."""
    A = R[:k, :k]
    Bk = R[:k, k:]
    C = R[k:, k:]
    Ainv = np.linalg.inv(A)
    U = Ainv @ Bk
    omega = 1.0 / np.linalg.norm(Ainv, axis=1)   # 1 / |row i of A_k^{-1}|
    gamma = np.linalg.norm(C, axis=0)             # |column j of C_k|
    rho = np.sqrt(U ** 2 + (gamma[None, :] / omega[:, None]) ** 2)
    return A, Bk, C, rho


def drrqr(M, k, f=2.0, max_swaps=1000):
    """M [rows, n] float64 -> (perm, rho_max, swaps): perm[:k] are the kept
    channels in selection order."""
    import scipy.linalg
    M = _as_f64(M)
    n = M.shape[1]
    _, _, perm = scipy.linalg.qr(M, mode="economic", pivoting=True)
    perm = np.array(perm)
    swaps = 0
    while True:
        R = scipy.linalg.qr(M[:, perm], mode="r")[0][:n, :n]
        _, _, _, rho = rrqr_factors(R, k)
        i, j = np.unravel_index(np.argmax(rho), rho.shape)
        if rho[i, j] <= f or swaps >= max_swaps:
            return perm, float(rho.max()), swaps
        perm[i], perm[k + j] = perm[k + j], perm[i]
        swaps += 1


def gather_normalize(x, idx, eps=1e-12):
    """x: [..., H, K_in]; idx: [H, K_out] integer channel indices.  Returns
    float64 [..., H, K_out]: the kept channels of each head, divided by their
    Euclidean norm (or by eps when that norm is smaller)."""
    x = _as_f64(x)
    idx = np.asarray(idx)
    H = x.shape[-2]
    assert idx.ndim == 2 and idx.shape[0] == H
    y = np.take_along_axis(x, np.broadcast_to(idx, x.shape[:-2] + idx.shape), axis=-1)
    n = np.sqrt(np.einsum("...k,...k->...", y, y))
    return y / np.maximum(n, eps)[..., None]
