"""Seeded synthetic inputs for the gated delta-rule workloads.

This module only draws random numbers and rounds them to the run dtype.  It
holds none of the recurrence's arithmetic, so both the GPU path and the CPU
oracle may consume its arrays: the oracle upcasts the exact rounded values to
float64, the GPU receives the same values as bf16 bits or fp32.

Workloads (shapes and value distributions follow the pages' models: per-head
states of 128 x 128, L2-normalised keys and queries, sigmoid write strengths,
input-dependent decay):

  tiny        B=1,  H=1,  T=256,   K=V=32,  fp32
  prefill     B=8,  H=16, T=4096,  K=V=128, bf16 q/k/v, chunk 64
  pruned      the prefill draws with q/k reduced to a fixed random per-head
              subset of 64 of the 128 key channels, re-normalised over the
              kept channels (state 128 x 64)
  decode      B=64 (or 1), H=16, V=128, K in {128, 64}, 1024 single-token
              steps from a low-stable-rank initial state
  long        B=1,  H=16, T=65536, K=V=128, bf16, alpha in [0.9995, 0.9999],
              keys in a narrow cone (|mean k| ~ 0.9 per head)
  gated       the prefill shapes under the channel-gated rules (KDA, GDN2):
              per-key-channel decay, and for GDN2 per-channel erase / write
              gates
  calibration key/query activations for channel selection: per-head
              channel scales and a shared low-rank channel mixing, then
              per-token L2 normalisation

Random streams: numpy PCG64.  The tiny workload uses seed ``seed`` directly;
the others use child ``i`` of ``SeedSequence(seed)`` (prefill and
pruned share child 1, so the pruned run sees the same Gaussian draws).  Draw
order inside a stream: q, k, v, beta logits, alpha logits, pruning subsets,
initial state.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

WORKLOADS = ("tiny", "prefill", "pruned", "decode", "long", "gated", "calibration")


def round_to_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 (ties to even); returns float32 holding the
    exactly representable values."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x32.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)  # finite inputs only: no overflow
    return r.view(np.float32)


def bf16_bits(x32: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    return (x32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _round(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError(dtype)


def _unit_rows(z: np.ndarray) -> np.ndarray:
    return z / np.linalg.norm(z, axis=-1, keepdims=True)


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _stream(seed: int, index: int) -> np.random.Generator:
    if index == 0:
        return np.random.default_rng(seed)
    children = np.random.SeedSequence(seed).spawn(max(5, index + 1))
    return np.random.Generator(np.random.PCG64(children[index]))


@dataclass
class Problem:
    """One batch of inputs.  Arrays are float32 holding values exact in
    ``dtype``; q/k are [B,T,H,K], v is [B,T,H,V], alpha/beta are [B,T,H],
    S0 is [B,H,V,K] or None."""

    name: str
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    S0: np.ndarray | None
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, T, H, K = self.k.shape
        return B, T, H, K, self.v.shape[-1]


def _gated_draws(rng, B, T, H, K, V):
    """Shared Gaussian draws for the prefill/pruned/decode recipes."""
    zq = rng.standard_normal((B, T, H, K))
    zk = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    beta = _sigmoid(rng.standard_normal((B, T, H)))
    # log alpha = -softplus(x), x ~ N(m_h, 0.5^2) around a per-head centre
    # m_h ~ N(-4, 1.5^2): gives per-head decay horizons from a few tokens to
    # about a thousand (the i.i.d.-per-token reading would give every head the
    # same ~20-token horizon).
    m_h = rng.normal(-4.0, 1.5, size=(H,))
    x = rng.normal(m_h[None, None, :], 0.5, size=(B, T, H))
    alpha = np.exp(-_softplus(x))
    return zq, zk, v, beta, alpha


def _prune_subsets(rng, H, K, Kp):
    idx = np.stack([np.sort(rng.permutation(K)[:Kp]) for _ in range(H)])
    return idx.astype(np.int32)


def make_tiny(seed=0, B=1, H=1, T=256, K=32, V=32, dtype="fp32") -> Problem:
    rng = _stream(seed, 0)
    q = _unit_rows(rng.standard_normal((B, T, H, K)))
    k = _unit_rows(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    beta = _sigmoid(rng.standard_normal((B, T, H)))
    alpha = np.exp(-_softplus(rng.normal(-3.0, 1.0, size=(B, T, H))))
    return Problem("tiny", dtype, _round(q, dtype), _round(k, dtype), _round(v, dtype),
                   alpha.astype(np.float32), beta.astype(np.float32), None,
                   {"seed": seed})


def make_prefill(seed=0, B=8, T=4096, H=16, K=128, V=128, dtype="bf16", pruned_K=None,
                 with_S0=False) -> Problem:
    """Gated DeltaNet layer prefill.  With ``pruned_K`` the same draws are
    gathered to a fixed random per-head channel subset and re-normalised."""
    rng = _stream(seed, 1)
    zq, zk, v, beta, alpha = _gated_draws(rng, B, T, H, K, V)
    meta = {"seed": seed}
    if pruned_K is not None:
        idx = _prune_subsets(rng, H, K, pruned_K)
        hh = np.arange(H)[:, None]
        zq = zq[:, :, hh, idx]
        zk = zk[:, :, hh, idx]
        meta["kept_channels"] = idx
    S0 = None
    if with_S0:
        Kc = zk.shape[-1]
        S0 = (0.1 * rng.standard_normal((B, H, V, Kc))).astype(np.float32)
    q = _round(_unit_rows(zq), dtype)
    k = _round(_unit_rows(zk), dtype)
    name = "pruned" if pruned_K is not None else "prefill"
    return Problem(name, dtype, q, k, _round(v, dtype), alpha.astype(np.float32),
                   beta.astype(np.float32), S0, meta)


def low_stable_rank_state(rng, B, H, V, K, terms=8, tail=1e-3) -> np.ndarray:
    """S0 = sum_i (1/i) a_i b_i^T + tail * G per head, a_i, b_i unit Gaussian
    directions, G ~ N(0,1) entrywise."""
    S = np.zeros((B, H, V, K))
    for i in range(1, terms + 1):
        a = _unit_rows(rng.standard_normal((B, H, V)))
        b = _unit_rows(rng.standard_normal((B, H, K)))
        S += (1.0 / i) * a[..., :, None] * b[..., None, :]
    S += tail * rng.standard_normal((B, H, V, K))
    return S.astype(np.float32)


def make_decode(seed=0, B=64, H=16, K=128, V=128, steps=1024, dtype="bf16",
                pruned_K=None) -> Problem:
    """Batched decode: ``steps`` single-token steps stored along the T axis
    ([B, steps, H, *]); step t uses q[:, t], k[:, t], ...  The initial state is
    low-stable-rank.  With ``pruned_K`` the keys/queries and the initial state
    keep the same fixed random per-head channel subset (S0' = S0 P_I^T)."""
    rng = _stream(seed, 3)
    zq, zk, v, beta, alpha = _gated_draws(rng, B, steps, H, K, V)
    meta = {"seed": seed, "steps": steps}
    idx = None
    if pruned_K is not None:
        idx = _prune_subsets(rng, H, K, pruned_K)
        hh = np.arange(H)[:, None]
        zq = zq[:, :, hh, idx]
        zk = zk[:, :, hh, idx]
        meta["kept_channels"] = idx
    S0 = low_stable_rank_state(rng, B, H, V, K)
    if idx is not None:
        S0 = np.ascontiguousarray(np.take_along_axis(S0, idx[None, :, None, :], axis=-1))
    q = _round(_unit_rows(zq), dtype)
    k = _round(_unit_rows(zk), dtype)
    return Problem("decode", dtype, q, k, _round(v, dtype), alpha.astype(np.float32),
                   beta.astype(np.float32), S0, meta)


CONE_OFFSET = 8.18  # |mu_h|: with noise 0.35 N(0, I_128) gives |mean k| ~ 0.90


def make_long(seed=0, B=1, T=65536, H=16, K=128, V=128, dtype="bf16") -> Problem:
    """Long-context prefill: long-horizon decay alpha ~ U[0.9995, 0.9999] per
    (t, h) and keys in a narrow per-head cone k = normalise(mu_h + 0.35 z)."""
    rng = _stream(seed, 4)
    q = _unit_rows(rng.standard_normal((B, T, H, K)))
    mu = CONE_OFFSET * _unit_rows(rng.standard_normal((H, K)))
    k = _unit_rows(mu[None, None] + 0.35 * rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    beta = _sigmoid(rng.standard_normal((B, T, H)))
    alpha = rng.uniform(0.9995, 0.9999, size=(B, T, H))
    return Problem("long", dtype, _round(q, dtype), _round(k, dtype), _round(v, dtype),
                   alpha.astype(np.float32), beta.astype(np.float32), None,
                   {"seed": seed, "cone_offset": CONE_OFFSET})


@dataclass
class GatedProblem:
    """Inputs of the channel-gated rules: q/k [B,T,H,K], v [B,T,H,V], alpha
    [B,T,H,K]; beta [B,T,H] for KDA, b [B,T,H,K] and w [B,T,H,V] for GDN2
    (the unused ones are None); S0 [B,H,V,K] or None."""

    gate: str
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray | None
    b: np.ndarray | None
    w: np.ndarray | None
    S0: np.ndarray | None
    meta: dict = field(default_factory=dict)


def make_channel_gated(seed=0, B=8, T=4096, H=16, K=128, V=128, dtype="bf16", gate="kda",
                       with_S0=False) -> GatedProblem:
    """q, k, v and beta drawn as the prefill workload; the decay per key
    channel, log alpha[t, h, c] = -softplus(x), x ~ N(m_{h,c}, 0.5^2) around
    a per-(head, channel) centre m_{h,c} ~ N(-4, 1.5^2) (the per-head centres
    of the prefill workload, one per channel); for GDN2 the erase gate
    b = sigmoid(N(0,1)) per key channel and the write gate w = sigmoid(N(0,1))
    per value channel, per token."""
    rng = _stream(seed, 5)
    zq, zk, v, beta, _ = _gated_draws(rng, B, T, H, K, V)
    m = rng.normal(-4.0, 1.5, size=(H, K))
    x = rng.normal(m[None, None], 0.5, size=(B, T, H, K))
    alpha = np.exp(-_softplus(x)).astype(np.float32)
    bg = wg = None
    if gate == "gdn2":
        bg = _sigmoid(rng.standard_normal((B, T, H, K))).astype(np.float32)
        wg = _sigmoid(rng.standard_normal((B, T, H, V))).astype(np.float32)
        beta = None
    elif gate != "kda":
        raise ValueError(gate)
    S0 = (0.1 * rng.standard_normal((B, H, V, K))).astype(np.float32) if with_S0 else None
    return GatedProblem(gate, dtype, _round(_unit_rows(zq), dtype), _round(_unit_rows(zk), dtype),
                        _round(v, dtype), alpha,
                        None if beta is None else beta.astype(np.float32), bg, wg, S0,
                        {"seed": seed})


def make_calibration(seed=0, B=8, T=4096, H=16, K=128, rank=16, dtype="bf16"):
    """Calibration activations (k, q) [B, T, H, K] for channel selection.
    Per head: channel scales s_c ~ LogNormal(0, 0.5^2) and a mixing
    L ~ N(0, 1/rank) of shape [K, rank] shared by keys and queries; a token is
    x = s (.) (g + 1.5 L w), g ~ N(0, I_K), w ~ N(0, I_rank), then L2-normalised,
    so that channels differ in energy and are correlated (the structure a
    channel selector has to see; i.i.d. channels would make every subset
    equivalent)."""
    rng = _stream(seed, 6)
    s = rng.lognormal(0.0, 0.5, size=(H, K))
    L = rng.standard_normal((H, K, rank)) / np.sqrt(rank)

    def draw():
        g = rng.standard_normal((B, T, H, K))
        w = rng.standard_normal((B, T, H, rank))
        x = s[None, None] * (g + 1.5 * np.einsum("hkr,bthr->bthk", L, w))
        return _round(_unit_rows(x), dtype)

    k = draw()
    q = draw()
    return k, q


def take_gated_sequences(p: GatedProblem, b_idx, h_idx) -> GatedProblem:
    """Sub-problem of sequences (b, h), b in b_idx, h in h_idx."""
    sl = np.ix_(np.asarray(b_idx), np.arange(p.k.shape[1]), np.asarray(h_idx))

    def g(x):
        return None if x is None else np.ascontiguousarray(x[sl])

    S0 = None if p.S0 is None else np.ascontiguousarray(p.S0[np.ix_(b_idx, h_idx)])
    return GatedProblem(p.gate, p.dtype, g(p.q), g(p.k), g(p.v), g(p.alpha), g(p.beta), g(p.b),
                        g(p.w), S0, dict(p.meta))


def take_sequences(p: Problem, b_idx, h_idx) -> Problem:
    """Sub-problem holding only sequences (b, h) for b in b_idx, h in h_idx
    (for sampled oracle checks at full size)."""
    b_idx = np.asarray(b_idx)
    h_idx = np.asarray(h_idx)
    sl = np.ix_(b_idx, np.arange(p.k.shape[1]), h_idx)

    def g(x):
        return np.ascontiguousarray(x[sl])

    S0 = None if p.S0 is None else np.ascontiguousarray(p.S0[np.ix_(b_idx, h_idx)])
    return Problem(p.name, p.dtype, g(p.q), g(p.k), g(p.v), g(p.alpha), g(p.beta), S0,
                   dict(p.meta))
