"""The debug build (-DGDN_BOUNDS_CHECK, libgdn_bounds.so): the prefill kernels
check every segment range, TMA box coordinate, key-side block offset and gate
or gathered-row offset they derive, and record a failure in the device status
instead of making the access.  On the small and ragged prefill shapes of the
parity tests (one-pass, two-pass, segment-parallel and gathering forms) every
check must pass (status GDN_OK) and the results must still match the oracle.

The debug library is loaded in a child process, so that this test process
keeps the release library."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))
import numpy as np, torch
import oracle
from gated_delta_rule_49_gb300 import binding, build, inputs
from gpu_util import problem_to_dev, rel_err, to_np
binding.load(build.build(bounds_check=True))
res = []

def run(p, ws_kind):
    B, T, H, K, V = p.shape
    d = problem_to_dev(p)
    o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ST = torch.full((B, H, V, K), float("nan"), device="cuda")
    need = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    if ws_kind == "two":
        need = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], o, ST, B, T, H,
                        K, V, binding.GDN_BF16, ws if need else None, need)
    st = binding.gdn_get_last_device_status()
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    res.append({"case": f"{ws_kind} B{B} T{T} H{H} K{K}", "status": st,
                "o": rel_err(to_np(o), o_ref), "S": rel_err(to_np(ST), S_ref)})

for K in (128, 64):
    for (B, T, H) in ((2, 300, 3), (1, 65, 1), (3, 1, 2), (4, 577, 8)):
        p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=T + K, with_S0=True)
        run(p, "one")
        run(p, "two")
    rng = np.random.default_rng(K)
    p = inputs.make_prefill(B=1, T=2113, H=2, K=K, seed=3, with_S0=True)  # segment-parallel
    run(p, "one")
    run(p, "two")

# the gathering form (full-width q / k, 64 kept channels)
rng = np.random.default_rng(1)
B, T, H = 2, 333, 3
r = inputs.round_to_bf16
qf = r(rng.standard_normal((B, T, H, 128)))
kf = r(rng.standard_normal((B, T, H, 128)))
v = r(rng.standard_normal((B, T, H, 128)))
al = rng.uniform(0.9, 1.0, size=(B, T, H)).astype(np.float32)
be = rng.uniform(0.0, 1.0, size=(B, T, H)).astype(np.float32)
idx = np.stack([np.sort(rng.permutation(128)[:64]) for _ in range(H)]).astype(np.int32)
bf = lambda x: torch.from_numpy(inputs.bf16_bits(np.ascontiguousarray(x, np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
o, ST = binding.prefill_gathered(bf(qf), bf(kf), torch.from_numpy(idx).cuda(), bf(v),
                                 torch.from_numpy(al).cuda(), torch.from_numpy(be).cuda())
st = binding.gdn_get_last_device_status()
o_ref, S_ref = oracle.recurrence(r(oracle.gather_normalize(qf, idx)),
                                 r(oracle.gather_normalize(kf, idx)), v, al, be)
res.append({"case": "gathered", "status": st, "o": rel_err(to_np(o), o_ref),
            "S": rel_err(to_np(ST), S_ref)})
print(json.dumps(res))
'''


def test_bounds_checked_build_passes_every_check():
    env = dict(os.environ)
    code = "import os\nROOT = " + repr(ROOT) + "\n" + CHILD
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    res = json.loads(out.stdout.strip().splitlines()[-1])
    assert len(res) == 21
    for r in res:
        assert r["status"] == 0, r
        assert r["o"] <= 1e-2 and r["S"] <= 1e-2, r
