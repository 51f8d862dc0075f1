"""Thin ctypes binding over libgdn.so (``include/gdn.h``).

Argument marshalling only: every step of the recurrence runs in the
library's CUDA kernels.  Functions with the C names take torch CUDA tensors
(or raw integer device pointers) for every buffer, pass ``data_ptr()`` and the
current torch stream, and raise ``GDNError`` on a negative status.  There is
no CPU fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_ALIGNMENT = -3
GDN_ERR_CUDA = -4
GDN_ERR_TIMEOUT = -5
GDN_ERR_WORKSPACE = -6
GDN_ERR_DEVICE_BOUNDS = -7
GDN_WARN_ZERO_STATE = 1
GDN_WARN_NOT_CONVERGED = 2
GDN_WARN_RANK_DEFICIENT = 3

GDN_BF16 = 0
GDN_FP32 = 1

GDN_GATE_SCALAR = 0
GDN_GATE_KDA = 1
GDN_GATE_GDN2 = 2
GATES = {"gdn": GDN_GATE_SCALAR, "kda": GDN_GATE_KDA, "gdn2": GDN_GATE_GDN2}

EXPORTS = (
    "gdn_prefill",
    "gdn_prefill_workspace_size",
    "gdn_prefill_two_pass_workspace_size",
    "gdn_decode_step",
    "gdn_state_rank",
    "gdn_get_last_device_status",
    "gdn_status_string",
    "gdn_version",
    "gdn_selftest_wait_timeout",
    "gdn_prefill_noalloc",
    "gdn_prefill_noalloc_max_workspace",
    "gdn_gather_normalize",
    "gdn_decode_step_gathered",
    "gdn_prefill_gated",
    "gdn_decode_step_gated",
    "gdn_state_truncate",
    "gdn_prefill_truncated",
    "gdn_channel_gram_workspace_size",
    "gdn_channel_gram",
    "gdn_drrqr_select",
    "gdn_prefill_host_workspace_size",
    "gdn_prefill_host",
    "gdn_prefill_gathered",
    "gdn_prefill_gathered_workspace_size",
    "gdn_prefill_gated_chunked",
    "gdn_prefill_gated_chunked_workspace_size",
)

_lock = threading.Lock()
_lib = None


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (built by ``gated_delta_rule_49_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libgdn.so is not built ({path} missing): run "
                "`python -m gated_delta_rule_49_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gdn_prefill.argtypes = [vp] * 8 + [i] * 6 + [vp, sz, vp]
        lib.gdn_prefill.restype = i
        lib.gdn_prefill_workspace_size.argtypes = [i] * 6
        lib.gdn_prefill_workspace_size.restype = sz
        lib.gdn_prefill_two_pass_workspace_size.argtypes = [i] * 6
        lib.gdn_prefill_two_pass_workspace_size.restype = sz
        lib.gdn_decode_step.argtypes = [vp] * 7 + [i] * 5 + [vp]
        lib.gdn_decode_step.restype = i
        lib.gdn_state_rank.argtypes = [vp, i, i, i, vp, vp, vp, i, f, vp]
        lib.gdn_state_rank.restype = i
        lib.gdn_get_last_device_status.argtypes = [vp]
        lib.gdn_get_last_device_status.restype = i
        lib.gdn_status_string.argtypes = [i]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = i
        lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
        lib.gdn_selftest_wait_timeout.restype = i
        lib.gdn_prefill_noalloc.argtypes = [vp] * 8 + [i] * 6 + [vp]
        lib.gdn_prefill_noalloc.restype = i
        lib.gdn_gather_normalize.argtypes = [vp, vp, vp, ctypes.c_longlong, i, i, i, i, vp]
        lib.gdn_gather_normalize.restype = i
        lib.gdn_decode_step_gathered.argtypes = [vp, vp, vp, i] + [vp] * 5 + [i] * 5 + [vp]
        lib.gdn_decode_step_gathered.restype = i
        lib.gdn_prefill_gated.argtypes = [vp] * 10 + [i] * 7 + [vp]
        lib.gdn_prefill_gated.restype = i
        lib.gdn_prefill_gated_chunked.argtypes = [vp] * 10 + [i] * 7 + [vp, sz, vp]
        lib.gdn_prefill_gated_chunked.restype = i
        lib.gdn_prefill_gated_chunked_workspace_size.argtypes = [i] * 7
        lib.gdn_prefill_gated_chunked_workspace_size.restype = sz
        lib.gdn_decode_step_gated.argtypes = [vp] * 9 + [i] * 6 + [vp]
        lib.gdn_decode_step_gated.restype = i
        lib.gdn_state_truncate.argtypes = [vp, i, i, i, i, vp, i, vp]
        lib.gdn_state_truncate.restype = i
        lib.gdn_prefill_truncated.argtypes = [vp] * 8 + [i] * 9 + [vp, sz, vp]
        lib.gdn_prefill_truncated.restype = i
        lib.gdn_channel_gram_workspace_size.argtypes = [i] * 4
        lib.gdn_channel_gram_workspace_size.restype = sz
        lib.gdn_channel_gram.argtypes = [vp, vp] + [i] * 5 + [vp, vp, sz, vp]
        lib.gdn_channel_gram.restype = i
        lib.gdn_drrqr_select.argtypes = [vp, i, i, i, f, i, vp, vp, vp, vp]
        lib.gdn_drrqr_select.restype = i
        lib.gdn_prefill_host_workspace_size.argtypes = [i] * 7
        lib.gdn_prefill_host_workspace_size.restype = sz
        lib.gdn_prefill_host.argtypes = [vp] * 8 + [i] * 7 + [vp, sz, vp]
        lib.gdn_prefill_host.restype = i
        lib.gdn_prefill_noalloc_max_workspace.argtypes = []
        lib.gdn_prefill_noalloc_max_workspace.restype = sz
        lib.gdn_prefill_gathered.argtypes = [vp, vp, vp, i] + [vp] * 6 + [i] * 6 + [vp, sz, vp]
        lib.gdn_prefill_gathered.restype = i
        lib.gdn_prefill_gathered_workspace_size.argtypes = [i] * 7
        lib.gdn_prefill_gathered_workspace_size.restype = sz
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().gdn_status_string(int(status)).decode()
    except RuntimeError:
        return "libgdn.so not loaded"


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_FP32
    raise GDNError(GDN_ERR_INVALID_ARG, f"dtype {t.dtype}")


def _check(status: int, where: str) -> int:
    if status < 0:
        raise GDNError(status, where)
    return status


def gdn_prefill(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V, dtype, workspace=None,
                workspace_bytes=0, stream=None) -> int:
    st = load().gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                            _ptr(o), _ptr(S_T), B, T, H, K, V, dtype, _ptr(workspace),
                            workspace_bytes, _stream(stream))
    return _check(st, "gdn_prefill")


def gdn_prefill_noalloc(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V, dtype,
                        stream=None) -> int:
    """gdn_prefill without a workspace argument: its scratch is a fixed array
    inside the library (for callers that cannot allocate device memory)."""
    st = load().gdn_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                                    _ptr(o), _ptr(S_T), B, T, H, K, V, dtype, _stream(stream))
    return _check(st, "gdn_prefill_noalloc")


def gdn_prefill_noalloc_max_workspace() -> int:
    return int(load().gdn_prefill_noalloc_max_workspace())


def gdn_prefill_workspace_size(B, T, H, K, V, dtype) -> int:
    return int(load().gdn_prefill_workspace_size(B, T, H, K, V, dtype))


def gdn_prefill_two_pass_workspace_size(B, T, H, K, V, dtype) -> int:
    return int(load().gdn_prefill_two_pass_workspace_size(B, T, H, K, V, dtype))


def gdn_decode_step(q, k, v, alpha, beta, S, o, B, H, K, V, dtype, stream=None) -> int:
    st = load().gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S),
                                _ptr(o), B, H, K, V, dtype, _stream(stream))
    return _check(st, "gdn_decode_step")


def gdn_state_rank(S, BH, V, K, fro2, sigma1, stable_rank, max_iter=500, tol=1e-7,
                   stream=None) -> int:
    st = load().gdn_state_rank(_ptr(S), BH, V, K, _ptr(fro2), _ptr(sigma1), _ptr(stable_rank),
                               max_iter, tol, _stream(stream))
    return _check(st, "gdn_state_rank")


def gdn_gather_normalize(x, idx, y, N, H, K_in, K_out, dtype, stream=None) -> int:
    st = load().gdn_gather_normalize(_ptr(x), _ptr(idx), _ptr(y), N, H, K_in, K_out, dtype,
                                     _stream(stream))
    return _check(st, "gdn_gather_normalize")


def gdn_decode_step_gathered(q_full, k_full, idx, K_in, v, alpha, beta, S, o, B, H, K, V, dtype,
                             stream=None) -> int:
    st = load().gdn_decode_step_gathered(_ptr(q_full), _ptr(k_full), _ptr(idx), K_in, _ptr(v),
                                         _ptr(alpha), _ptr(beta), _ptr(S), _ptr(o), B, H, K, V,
                                         dtype, _stream(stream))
    return _check(st, "gdn_decode_step_gathered")


def gdn_prefill_gated(q, k, v, alpha, beta, b, w, S0, o, S_T, B, T, H, K, V, gate, dtype,
                      stream=None) -> int:
    st = load().gdn_prefill_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(b),
                                  _ptr(w), _ptr(S0), _ptr(o), _ptr(S_T), B, T, H, K, V, gate,
                                  dtype, _stream(stream))
    return _check(st, "gdn_prefill_gated")


def gdn_prefill_gated_chunked(q, k, v, alpha, beta, b, w, S0, o, S_T, B, T, H, K, V, gate,
                              dtype, workspace, workspace_bytes, stream=None) -> int:
    st = load().gdn_prefill_gated_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                          _ptr(b), _ptr(w), _ptr(S0), _ptr(o), _ptr(S_T), B, T,
                                          H, K, V, gate, dtype, _ptr(workspace), workspace_bytes,
                                          _stream(stream))
    return _check(st, "gdn_prefill_gated_chunked")


def gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, gate, dtype) -> int:
    return load().gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, gate, dtype)


def prefill_gated_chunked(q, k, v, alpha, beta=None, b=None, w=None, S0=None, gate="kda",
                          want_o=True, want_state=True, workspace=None, stream=None):
    """gdn_prefill_gated_chunked on torch CUDA tensors (gate "kda" or "gdn2",
    K = V = 128, bf16); allocates the workspace unless one is given.
    Returns (o, S_T)."""
    import torch
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = torch.empty((B, T, H, V), dtype=v.dtype, device=v.device) if want_o else None
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device=v.device) if want_state else None
    need = gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, GATES[gate], _dtype_code(v))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=v.device)
    gdn_prefill_gated_chunked(q, k, v, alpha, beta, b, w, S0, o, ST, B, T, H, K, V, GATES[gate],
                              _dtype_code(v), workspace, workspace.numel(), stream)
    return o, ST


def gdn_decode_step_gated(q, k, v, alpha, beta, b, w, S, o, B, H, K, V, gate, dtype,
                          stream=None) -> int:
    st = load().gdn_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                      _ptr(b), _ptr(w), _ptr(S), _ptr(o), B, H, K, V, gate, dtype,
                                      _stream(stream))
    return _check(st, "gdn_decode_step_gated")


def prefill_gated(q, k, v, alpha, beta=None, b=None, w=None, S0=None, gate="kda",
                  want_o=True, want_state=True, stream=None):
    """gdn_prefill_gated on torch CUDA tensors: q, k [B,T,H,K]; v [B,T,H,V];
    alpha [B,T,H] (gate "gdn") or [B,T,H,K]; beta [B,T,H] ("gdn", "kda");
    b [B,T,H,K], w [B,T,H,V] ("gdn2").  Returns (o, S_T)."""
    import torch
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = torch.empty((B, T, H, V), dtype=v.dtype, device=v.device) if want_o else None
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device=v.device) if want_state else None
    gdn_prefill_gated(q, k, v, alpha, beta, b, w, S0, o, ST, B, T, H, K, V, GATES[gate],
                      _dtype_code(v), stream)
    return o, ST


def gdn_state_truncate(S, BH, V, K, r, sigma=None, max_sweeps=30, stream=None) -> int:
    st = load().gdn_state_truncate(_ptr(S), BH, V, K, r, _ptr(sigma), max_sweeps,
                                   _stream(stream))
    return _check(st, "gdn_state_truncate")


def gdn_prefill_truncated(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V, dtype, seg_len, r,
                          max_sweeps=30, workspace=None, workspace_bytes=0, stream=None) -> int:
    st = load().gdn_prefill_truncated(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                      _ptr(S0), _ptr(o), _ptr(S_T), B, T, H, K, V, dtype,
                                      seg_len, r, max_sweeps, _ptr(workspace), workspace_bytes,
                                      _stream(stream))
    return _check(st, "gdn_prefill_truncated")


def state_truncate(S, r, want_sigma=False, max_sweeps=30, stream=None):
    """In-place rank-r truncation of S [..., V, K] (float32 CUDA); returns the
    singular values [..., min(V, K)] if asked."""
    import torch
    V, K = S.shape[-2:]
    BH = S.numel() // (V * K)
    sigma = (torch.empty(S.shape[:-2] + (min(V, K),), dtype=torch.float32, device=S.device)
             if want_sigma else None)
    gdn_state_truncate(S, BH, V, K, r, sigma, max_sweeps, stream)
    return sigma


def prefill_truncated(q, k, v, alpha, beta, S0=None, seg_len=256, r=32, max_sweeps=30,
                      stream=None):
    """gdn_prefill_truncated on torch CUDA tensors.  Returns (o, S_T)."""
    import torch
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = torch.empty((B, T, H, V), dtype=v.dtype, device=v.device)
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device=v.device)
    dt = _dtype_code(v)
    L = min(seg_len, T) if T > 0 else 0
    need = max([gdn_prefill_workspace_size(B, n, H, K, V, dt) for n in (L, T % seg_len) if n] + [0])
    ws = torch.empty(need, dtype=torch.uint8, device=v.device) if need else None
    gdn_prefill_truncated(q, k, v, alpha, beta, S0, o, ST, B, T, H, K, V, dt, seg_len, r,
                          max_sweeps, ws, need, stream)
    return o, ST


def gdn_channel_gram_workspace_size(B, T, H, K) -> int:
    return int(load().gdn_channel_gram_workspace_size(B, T, H, K))


def gdn_channel_gram(k, q, B, T, H, K, dtype, G, workspace, workspace_bytes,
                     stream=None) -> int:
    st = load().gdn_channel_gram(_ptr(k), _ptr(q), B, T, H, K, dtype, _ptr(G), _ptr(workspace),
                                 workspace_bytes, _stream(stream))
    return _check(st, "gdn_channel_gram")


def gdn_drrqr_select(G, H, n, k, f, max_swaps, idx, rho_max=None, swaps=None,
                     stream=None) -> int:
    st = load().gdn_drrqr_select(_ptr(G), H, n, k, ctypes.c_float(f), max_swaps, _ptr(idx),
                                 _ptr(rho_max), _ptr(swaps), _stream(stream))
    return _check(st, "gdn_drrqr_select")


def channel_gram(k, q, stream=None):
    """k, q [B, T, H, 128] bf16 CUDA -> G [H, 128, 128] float32."""
    import torch
    B, T, H, K = k.shape
    G = torch.empty((H, K, K), dtype=torch.float32, device=k.device)
    need = gdn_channel_gram_workspace_size(B, T, H, K)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=k.device)
    gdn_channel_gram(k, q, B, T, H, K, _dtype_code(k), G, ws, need, stream)
    return G


def drrqr_select(G, k, f=2.0, max_swaps=1000, stream=None):
    """G [H, n, n] float32 CUDA -> (idx [H, k] int32 in selection order,
    rho_max [H], swaps [H])."""
    import torch
    H, n, _ = G.shape
    idx = torch.empty((H, k), dtype=torch.int32, device=G.device)
    rho = torch.empty(H, dtype=torch.float32, device=G.device)
    sw = torch.empty(H, dtype=torch.int32, device=G.device)
    gdn_drrqr_select(G, H, n, k, f, max_swaps, idx, rho, sw, stream)
    return idx, rho, sw


def gdn_prefill_host_workspace_size(B, T, H, K, V, dtype, window) -> int:
    return int(load().gdn_prefill_host_workspace_size(B, T, H, K, V, dtype, window))


def gdn_prefill_host(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V, dtype, window, workspace,
                     workspace_bytes, stream=None) -> int:
    """Host-buffer prefill: q .. S_T are (pinned) CPU tensors or host addresses;
    workspace is device memory."""
    st = load().gdn_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                                 _ptr(o), _ptr(S_T), B, T, H, K, V, dtype, window,
                                 _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(st, "gdn_prefill_host")


def gdn_prefill_gathered_workspace_size(B, T, H, K_in, K, V, dtype) -> int:
    return int(load().gdn_prefill_gathered_workspace_size(B, T, H, K_in, K, V, dtype))


def gdn_prefill_gathered(q_full, k_full, idx, K_in, v, alpha, beta, S0, o, S_T, B, T, H, K, V,
                         dtype, workspace, workspace_bytes, stream=None) -> int:
    st = load().gdn_prefill_gathered(_ptr(q_full), _ptr(k_full), _ptr(idx), K_in, _ptr(v),
                                     _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(o), _ptr(S_T), B, T,
                                     H, K, V, dtype, _ptr(workspace), workspace_bytes,
                                     _stream(stream))
    return _check(st, "gdn_prefill_gathered")


def prefill_gathered(q_full, k_full, idx, v, alpha, beta, S0=None, want_o=True, want_state=True,
                     stream=None):
    """The pruned prefill from full-width q / k ([B, T, H, 128] bf16) and the kept
    channels idx ([H, 64] int32): returns (o, S_T) with S_T [B, H, 128, 64]."""
    import torch
    B, T, H, K_in = k_full.shape
    K, V = idx.shape[1], v.shape[-1]
    dt = _dtype_code(k_full)
    o = torch.empty((B, T, H, V), dtype=v.dtype, device=v.device) if want_o else None
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device=v.device) if want_state else None
    need = gdn_prefill_gathered_workspace_size(B, T, H, K_in, K, V, dt)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=v.device)
    gdn_prefill_gathered(q_full, k_full, idx, K_in, v, alpha, beta, S0, o, ST, B, T, H, K, V, dt,
                         ws, need, stream)
    return o, ST


def gather_normalize(x, idx, stream=None):
    """x [..., H, K_in] (bf16/fp32 CUDA); idx [H, K_out] int32 CUDA.  Returns
    the pruned, renormalised [..., H, K_out]."""
    import torch
    H, K_in = x.shape[-2:]
    K_out = idx.shape[-1]
    N = x.numel() // (H * K_in)
    y = torch.empty(x.shape[:-1] + (K_out,), dtype=x.dtype, device=x.device)
    gdn_gather_normalize(x, idx, y, N, H, K_in, K_out, _dtype_code(x), stream)
    return y


def gdn_get_last_device_status(stream=None) -> int:
    return int(load().gdn_get_last_device_status(_stream(stream)))


def gdn_status_string(status: int) -> str:
    return status_string(status)


def gdn_selftest_wait_timeout(limit_cycles, stream=None) -> int:
    st = load().gdn_selftest_wait_timeout(int(limit_cycles), _stream(stream))
    return _check(st, "gdn_selftest_wait_timeout")


def gdn_version() -> int:
    return int(load().gdn_version())


# ---- tensor-level conveniences (allocate outputs with torch, then call) ----

def prefill(q, k, v, alpha, beta, S0=None, want_o=True, want_state=True, out_state=None,
            stream=None, two_pass=True):
    """q, k [B,T,H,K]; v [B,T,H,V] (bf16 or fp32 CUDA tensors); alpha, beta
    [B,T,H] fp32; S0 [B,H,V,K] fp32 or None.  Returns (o, S_T).  two_pass:
    allocate the workspace of the two-pass form where the problem has one
    (identical results; False runs the one-pass form)."""
    import torch
    B, T, H, K = k.shape
    V = v.shape[-1]
    dt = _dtype_code(k)
    o = torch.empty((B, T, H, V), dtype=k.dtype, device=k.device) if want_o else None
    ST = None
    if want_state:
        ST = out_state if out_state is not None else torch.empty(
            (B, H, V, K), dtype=torch.float32, device=k.device)
    ws_bytes = gdn_prefill_workspace_size(B, T, H, K, V, dt)
    if two_pass:
        ws_bytes = max(ws_bytes, gdn_prefill_two_pass_workspace_size(B, T, H, K, V, dt))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=k.device) if ws_bytes else None
    gdn_prefill(q, k, v, alpha, beta, S0, o, ST, B, T, H, K, V, dt, ws, ws_bytes, stream)
    return o, ST


def decode_step(q, k, v, alpha, beta, S, o=None, stream=None):
    """One token: q, k [B,H,K]; v [B,H,V]; alpha, beta [B,H]; S [B,H,V,K]
    updated in place.  Returns o [B,H,V]."""
    import torch
    B, H, K = k.shape
    V = v.shape[-1]
    if o is None:
        o = torch.empty((B, H, V), dtype=k.dtype, device=k.device)
    gdn_decode_step(q, k, v, alpha, beta, S, o, B, H, K, V, _dtype_code(k), stream)
    return o


def state_rank(S, max_iter=500, tol=1e-7, stream=None):
    """S [..., V, K] fp32.  Returns (fro2, sigma1, stable_rank) shaped [...]."""
    import torch
    lead = S.shape[:-2]
    V, K = S.shape[-2:]
    BH = 1
    for d in lead:
        BH *= d
    outs = [torch.empty(lead, dtype=torch.float32, device=S.device) for _ in range(3)]
    gdn_state_rank(S, BH, V, K, *outs, max_iter=max_iter, tol=tol, stream=stream)
    return tuple(outs)
