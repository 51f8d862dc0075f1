"""Helpers shared by the GPU parity tests: move generator arrays to the
device, run the library through its C ABI binding, and measure errors the way
the tolerances are stated (max |x_gpu - x_ref| / max |x_ref| per tensor)."""
import numpy as np

# Tolerances of the parity bar: bf16 q/k/v with a float32 state, and all-fp32.
TOL = {"bf16": 1e-2, "fp32": 1e-4}


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / den)


def to_dev(x, dtype, device="cuda"):
    """float32 array holding values exact in ``dtype`` -> torch CUDA tensor."""
    import torch
    from gated_delta_rule_49_gb300 import inputs
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return torch.from_numpy(inputs.bf16_bits(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(x).to(device)


def problem_to_dev(p):
    import torch
    d = {
        "q": to_dev(p.q, p.dtype), "k": to_dev(p.k, p.dtype), "v": to_dev(p.v, p.dtype),
        "alpha": torch.from_numpy(np.ascontiguousarray(p.alpha)).cuda(),
        "beta": torch.from_numpy(np.ascontiguousarray(p.beta)).cuda(),
        "S0": None if p.S0 is None else torch.from_numpy(np.ascontiguousarray(p.S0)).cuda(),
    }
    return d


def to_np(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def run_prefill(p, **kw):
    from gated_delta_rule_49_gb300 import binding
    d = problem_to_dev(p)
    o, ST = binding.prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], **kw)
    return (None if o is None else to_np(o)), (None if ST is None else to_np(ST))


def run_decode(p, steps=None):
    """Run p's T axis as successive decode steps through gdn_decode_step."""
    import torch
    from gated_delta_rule_49_gb300 import binding
    d = problem_to_dev(p)
    B, T, H, K = p.k.shape
    V = p.v.shape[-1]
    steps = T if steps is None else steps
    S = d["S0"].clone() if d["S0"] is not None else torch.zeros((B, H, V, K), device="cuda")
    outs = []
    for t in range(steps):
        o = binding.decode_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                d["v"][:, t].contiguous(), d["alpha"][:, t].contiguous(),
                                d["beta"][:, t].contiguous(), S)
        outs.append(o)
    o = torch.stack(outs, dim=1)
    return to_np(o), to_np(S)
