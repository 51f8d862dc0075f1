"""Benchmark of the gated delta-rule path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: Gated DeltaNet layer prefill, B=8, T=4096, H=16,
d_k = d_v = 128, bf16 q/k/v, fp32 state, chunk 64, S0 = 0.  A timed step is
one gdn_prefill call over the whole batch, given the two-pass workspace (a
key-side kernel over every chunk, then the state kernel: two launches per
step); `value` is tokens/s (B*T per step, summed over ranks) and `one_pass`
times the same call without the workspace (one fused kernel, identical
results).  The same JSON line carries the rest of the metric, measured in the
same run: the channel-pruned d_k' = 64 prefill and its speed-up, the decode
state GB/s (B = 64 and B = 1, d_k 128 and 64; as specified and L2-cold) and
the stable-rank epilogue time, plus one entry per further path (prologue,
truncation, DRRQR, long context, KDA/GDN2, fp32).  The roofline counts the
algorithmic bytes of the call against the time of both kernels; its traffic
is the two kernels' DRAM bytes from the committed ncu summary.

Inputs live in HBM before the timed region; the prefill working set
(q, k, v, o: 537 MB) is larger than L2, so no flush is needed between steps.
Multi-GPU (torchrun): every rank runs the same independent batch on its own
GPU (sequences shard with no exchange step); barrier + max over ranks.

--impl reference times the float64 CPU oracle (the reference arm of this
repository) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = {"workload": "gated-deltanet-prefill", "B": 8, "T": 4096, "H": 16, "d_k": 128,
            "d_v": 128, "chunk": 64, "state": "fp32", "qkv": "bf16", "S0": "zero"}
METRIC = "prefill tokens/s and decode state GB/s (% of HBM/TC roofline) at d_k 128 vs 64"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- accounting
def prefill_bytes(B, T, H, K, V, qkv_bytes=2, with_S0=False):
    """Algorithmic HBM bytes of one prefill launch: q, k, v read, o written,
    alpha/beta read, final state written (and S0 read if given)."""
    per_token_head = 2 * K * qkv_bytes + V * qkv_bytes + V * qkv_bytes + 8
    state = 4 * V * K * (2 if with_S0 else 1)
    return B * T * H * per_token_head + B * H * state


def prefill_flops(B, T, H, K, V, C=64):
    """Chunked-form FLOPs per launch: 2 * (3CK + 2CV + 3KV + C^2/6) per token-head
    (KK^T, W, QK^T; U~, P U; W S^T, Q S^T, state update; triangular solve)."""
    macs = 3 * C * K + 2 * C * V + 3 * K * V + C * C / 6.0
    return 2.0 * macs * B * T * H


def measured_traffic(profile, source):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source has changed since the counters were taken (the summary
    records the first 16 hex digits of the source's sha256)."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        src = open(os.path.join(ROOT, "gated_delta_rule_49_gb300", "csrc", source), "rb").read()
    except OSError:
        return None
    sha = re.search(r"sha256 \(first 16 hex\): `([0-9a-f]{16})`", text)
    byts = re.search(r"traffic_bytes_per_launch: (\d+)", text)
    if not sha or not byts or hashlib.sha256(src).hexdigest()[:16] != sha.group(1):
        return None
    return int(byts.group(1))


def decode_state_bytes(B, H, K, V):
    return 2 * 4 * V * K * B * H


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                clk, mx, util = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            smax = mx
            if util > 0:
                sm.append(clk)
            for n, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                    "samples": len(self.lines)}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples_under_load": len(sm)}


# ----------------------------------------------------------------- helpers
def to_dev_bf16(x, torch):
    from gated_delta_rule_49_gb300 import inputs
    bits = inputs.bf16_bits(np.ascontiguousarray(x, np.float32)).view(np.int16)
    return torch.from_numpy(bits).view(torch.bfloat16).cuda()


def problem_to_dev(p, torch):
    return dict(q=to_dev_bf16(p.q, torch), k=to_dev_bf16(p.k, torch), v=to_dev_bf16(p.v, torch),
                alpha=torch.from_numpy(np.ascontiguousarray(p.alpha)).cuda(),
                beta=torch.from_numpy(np.ascontiguousarray(p.beta)).cuda())


def time_calls(fn, steps, warmup, torch, barrier=None):
    """Warm up, then time exactly `steps` calls with CUDA events on the current
    stream; returns (total_ms, per-call ms list)."""
    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(steps):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return evs[0].elapsed_time(evs[-1]), per


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, barrier, max_over_ranks):
    import torch
    from gated_delta_rule_49_gb300 import binding, inputs

    binding.load()
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sampler = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
                           if "CUDA_VISIBLE_DEVICES" in os.environ else torch.cuda.current_device())
    sampler.start()
    launches = 0

    # ---- headline: prefill, d_k = 128 ----
    W = WORKLOAD
    B, T, H, K, V = W["B"], W["T"], W["H"], W["d_k"], W["d_v"]
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, V=V)
    d = problem_to_dev(p, torch)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device="cuda")
    # two-pass form: the workspace holds every chunk's key-side operands
    wsb = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def step():
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, ws, wsb)

    total_ms, per = time_calls(step, args.steps, args.warmup, torch, barrier)
    launches += 2 * args.steps  # key-side pass + state pass
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    tokens = B * T * world * args.steps
    value = tokens / (total_ms / 1e3)
    kern_ms = statistics.mean(per)
    byts = prefill_bytes(B, T, H, K, V)
    flops = prefill_flops(B, T, H, K, V)
    achieved_gbs = byts / (kern_ms / 1e3) / 1e9
    achieved_tf = flops / (kern_ms / 1e3) / 1e12
    status = binding.gdn_get_last_device_status()

    extra = {}
    # the one-pass form (no workspace) on the same inputs, for comparison
    if not args.quick:
        def step1():
            binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T,
                                H, K, V, binding.GDN_BF16)

        t1, _ = time_calls(step1, args.steps, args.warmup, torch, barrier)
        t1 = max_over_ranks(t1)
        extra["one_pass"] = {"ms_per_step": t1 / args.steps,
                             "tokens_per_s": B * T * world * args.steps / (t1 / 1e3),
                             "two_pass_speedup": t1 / total_ms, "launches": args.steps,
                             "note": "gdn_prefill without the two-pass workspace (one fused "
                                     "kernel); identical results"}
    SECTIONS = ("pruned", "prologue", "state_rank", "truncation", "drrqr", "long_context",
                "gated", "fp32", "decode")

    def want(name):
        return not args.quick and (args.only is None or args.only == name)

    if want("pruned") or want("prologue"):
        # ---- pruned d_k' = 64, same draws ----
        pp = inputs.make_prefill(B=B, T=T, H=H, K=K, V=V, pruned_K=64)
        dp = problem_to_dev(pp, torch)
        STp = torch.empty((B, H, V, 64), dtype=torch.float32, device="cuda")
        wsb64 = binding.gdn_prefill_two_pass_workspace_size(B, T, H, 64, V, binding.GDN_BF16)

        def step64():
            binding.gdn_prefill(dp["q"], dp["k"], dp["v"], dp["alpha"], dp["beta"], None, o, STp,
                                B, T, H, 64, V, binding.GDN_BF16, ws, wsb64)

        if want("pruned"):
            t64, per64 = time_calls(step64, args.steps, args.warmup, torch, barrier)
            t64 = max_over_ranks(t64)
            k64 = statistics.mean(per64)
            extra["pruned_dk64"] = {
                "tokens_per_s": B * T * world * args.steps / (t64 / 1e3),
                "ms_per_step": t64 / args.steps,
                "speedup_vs_dk128": (total_ms / args.steps) / (t64 / args.steps),
                "achieved_gbs": prefill_bytes(B, T, H, 64, V) / (k64 / 1e3) / 1e9,
                "achieved_tflops": prefill_flops(B, T, H, 64, V) / (k64 / 1e3) / 1e12,
            }
            extra["pruned_dk64"]["hbm_frac"] = (extra["pruned_dk64"]["achieved_gbs"] /
                                                peaks["hbm_gbs"])

        # ---- pruning prologue from the full-width q/k of the headline run ----
        if want("prologue"):
            idx = torch.from_numpy(pp.meta["kept_channels"].astype(np.int32)).cuda()
            extra["prologue"] = bench_prologue(args, torch, binding, d, idx, dp, o, peaks,
                                               barrier, max_over_ranks, world)
        del dp, pp

    # ---- stable-rank epilogue on the final states of the headline run ----
    if want("state_rank"):
        f2 = torch.empty(B * H, device="cuda")
        s1 = torch.empty_like(f2)
        er = torch.empty_like(f2)

        def rank_call():
            binding.gdn_state_rank(ST, B * H, V, K, f2, s1, er, 500, 1e-7)

        tr, perr = time_calls(rank_call, 5, 2, torch, barrier)
        extra["state_rank"] = {"ms_per_call": tr / 5, "states": B * H,
                               "median_er": float(er.median().item())}

    # ---- rank-r truncation: the headline's final states, and the segmented prefill ----
    if want("truncation"):
        extra["truncation"] = bench_truncation(args, torch, binding, d, ST, barrier,
                                               max_over_ranks, world)

    # ---- DRRQR channel selection (calibration Gram + selection) ----
    if want("drrqr"):
        extra["drrqr"] = bench_drrqr(args, torch, binding, inputs, peaks, barrier,
                                     max_over_ranks)

    # ---- long-context prefill: B=1, T=65536, H=16 (segment-parallel) ----
    if want("long_context"):
        extra["long_context"] = bench_long(args, torch, binding, inputs, peaks, barrier,
                                           max_over_ranks, world)

    # ---- channel-gated rules (KDA, GDN2) on the prefill shapes ----
    if want("gated"):
        extra["gated"] = bench_gated(args, torch, binding, inputs, peaks, barrier,
                                     max_over_ranks, world)

    # ---- all-fp32 mode on the prefill shapes ----
    if want("fp32"):
        extra["fp32"] = bench_fp32(args, torch, binding, inputs, peaks, barrier, max_over_ranks,
                                   world)

    # ---- decode: B = 64 and 1, d_k 128 and 64 ----
    if want("decode"):
        extra["decode"] = bench_decode(args, torch, binding, inputs, peaks, props, barrier,
                                       max_over_ranks)
    assert args.only is None or args.only in SECTIONS

    clocks = sampler.stop()

    # ---- end to end through the C ABI with host buffers ----
    e2e = bench_e2e(p, torch, binding, args, barrier, max_over_ranks, world)

    roof_bound = "hbm" if byts / peaks["hbm_gbs"] >= flops / 1e3 / peaks["bf16_tflops"] else "tensor"
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded generator; per-head decay centres, L2-normalised q/k)",
        "config": headline_config(W, world),
        "roofline": {
            "bound": roof_bound,
            "achieved": achieved_gbs if roof_bound == "hbm" else achieved_tf,
            "peak": peaks["hbm_gbs"] if roof_bound == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if roof_bound == "hbm" else "TFLOP/s",
            "frac": (achieved_gbs / peaks["hbm_gbs"]) if roof_bound == "hbm"
            else achieved_tf / peaks["bf16_tflops"],
            "traffic": measured_traffic("prefill_two_pass_d128_prefill-workload.md",
                                        "gdn_prefill_tc.cu"),
            "kernel": "gdn_prefill (two-pass: prefill_prep_kernel + prefill_state_kernel)",
            "algorithmic_bytes": byts,
            "algorithmic_flops": flops,
            "tensor_frac": achieved_tf / peaks["bf16_tflops"],
            "peak_source": peaks["source"],
        },
        "gpu_launches": launches,
        "device_status": status,
        "clocks": clocks,
        "e2e": e2e,
        "gpu": props.name,
        "sm_count": props.multi_processor_count,
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, seqs=args.cpu_seqs)
    return line


def bench_decode(args, torch, binding, inputs, peaks, props, barrier, max_over_ranks):
    """Decode state GB/s.  Steps are replayed from a CUDA graph; 'as specified'
    runs 64 steps on one state updated in place (it may sit in L2); 'l2_cold'
    rotates every step to the next of n state buffers with n * state >= 4x L2,
    and its graph holds max(64, n) steps so that every buffer is touched once
    per replay (the per-step inputs cycle over 64 drawn steps).  At B = 1 a
    step is latency-bound and only the as-specified run is reported.  At
    B = 64 the pruned step is also timed from full-width q/k: gathered and
    renormalised inside the step ('gathered'), and as two prologue launches
    followed by the plain step ('unfused')."""
    res = {}
    l2 = props.L2_cache_size if hasattr(props, "L2_cache_size") else 126 * 2**20
    H, V = 16, 128
    nsteps = 64
    launches = 0

    def steps_first(x, bf16=True):
        x = np.ascontiguousarray(np.moveaxis(x, 1, 0))
        return to_dev_bf16(x, torch) if bf16 else torch.from_numpy(x).cuda()

    def graph_time(call, S0, nbuf, B, K, per_step_launches):
        nonlocal launches
        gsteps = max(nsteps, nbuf)
        states = [S0.clone() for _ in range(nbuf)]
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for t in range(3):  # warm-up outside capture
                call(t, states[t % nbuf])
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for t in range(gsteps):
                call(t % nsteps, states[t % nbuf])
        reps = max(3, args.decode_reps)
        tot, _ = time_calls(g.replay, reps, 3, torch, barrier)
        launches += reps * gsteps * per_step_launches
        tot = max_over_ranks(tot)
        step_us = tot / reps / gsteps * 1e3
        gbs = decode_state_bytes(B, H, K, V) / (step_us / 1e6) / 1e9
        del g, states
        return {"us_per_step": step_us, "state_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                "state_buffers": nbuf, "graph_steps": gsteps,
                "tokens_per_s": B / (step_us / 1e6)}

    for B in (64, 1):
        for K in (128, 64):
            p = inputs.make_decode(B=B, H=H, K=128, V=V, steps=nsteps,
                                   pruned_K=None if K == 128 else 64)
            q, k, v = steps_first(p.q), steps_first(p.k), steps_first(p.v)
            al, be = steps_first(p.alpha, False), steps_first(p.beta, False)
            o = torch.empty((nsteps, B, H, V), dtype=torch.bfloat16, device="cuda")
            sbytes = 4 * B * H * V * K
            nbuf_cold = max(1, -(-4 * l2 // sbytes))
            S0 = torch.from_numpy(p.S0).cuda()
            modes = [("as_specified", 1)]
            if B > 1:  # a B = 1 step (1 MB of state) is latency-bound; no L2-cold run
                modes.append(("l2_cold", nbuf_cold))

            def plain(i, S):
                binding.gdn_decode_step(q[i], k[i], v[i], al[i], be[i], S, o[i], B, H, K, V,
                                        binding.GDN_BF16)

            res[f"B{B}_dk{K}"] = {m: graph_time(plain, S0, n, B, K, 1) for m, n in modes}
            if B == 64 and K == 64:
                pf = inputs.make_decode(B=B, H=H, K=128, V=V, steps=nsteps)
                qf, kf = steps_first(pf.q), steps_first(pf.k)
                idx = torch.from_numpy(p.meta["kept_channels"].astype(np.int32)).cuda()
                qg = torch.empty((B, H, K), dtype=torch.bfloat16, device="cuda")
                kg = torch.empty_like(qg)

                def fused(i, S):
                    binding.gdn_decode_step_gathered(qf[i], kf[i], idx, 128, v[i], al[i], be[i],
                                                     S, o[i], B, H, K, V, binding.GDN_BF16)

                def unfused(i, S):
                    binding.gdn_gather_normalize(qf[i], idx, qg, B, H, 128, K, binding.GDN_BF16)
                    binding.gdn_gather_normalize(kf[i], idx, kg, B, H, 128, K, binding.GDN_BF16)
                    binding.gdn_decode_step(qg, kg, v[i], al[i], be[i], S, o[i], B, H, K, V,
                                            binding.GDN_BF16)

                res[f"B{B}_dk{K}_gathered"] = {m: graph_time(fused, S0, n, B, K, 1)
                                               for m, n in modes}
                res[f"B{B}_dk{K}_unfused"] = {m: graph_time(unfused, S0, n, B, K, 3)
                                              for m, n in modes}
                del pf, qf, kf
            if B == 64 and K == 128:
                for gate in ("kda", "gdn2"):
                    pg = inputs.make_channel_gated(B=B, T=nsteps, H=H, K=K, V=V, gate=gate)
                    gq, gk, gv = steps_first(pg.q), steps_first(pg.k), steps_first(pg.v)
                    ga = steps_first(pg.alpha, False)
                    gb = None if pg.beta is None else steps_first(pg.beta, False)
                    gbb = None if pg.b is None else steps_first(pg.b, False)
                    gw = None if pg.w is None else steps_first(pg.w, False)
                    code = binding.GATES[gate]

                    def gated(i, S, gq=gq, gk=gk, gv=gv, ga=ga, gb=gb, gbb=gbb, gw=gw,
                              code=code):
                        binding.gdn_decode_step_gated(
                            gq[i], gk[i], gv[i], ga[i], None if gb is None else gb[i],
                            None if gbb is None else gbb[i], None if gw is None else gw[i], S,
                            o[i], B, H, K, V, code, binding.GDN_BF16)

                    res[f"B{B}_dk{K}_{gate}"] = {m: graph_time(gated, S0, n, B, K, 1)
                                                 for m, n in modes}
                    del pg, gq, gk, gv, ga, gb, gbb, gw
    for B in (64, 1):
        a, b = res[f"B{B}_dk128"], res[f"B{B}_dk64"]
        res[f"B{B}_speedup_dk64"] = {m: a[m]["us_per_step"] / b[m]["us_per_step"] for m in a}
    a, g = res["B64_dk128"], res["B64_dk64_gathered"]
    res["B64_speedup_dk64_gathered"] = {m: a[m]["us_per_step"] / g[m]["us_per_step"] for m in a}
    res["note"] = ("state GB/s = 8 V K B H / step time; steps replayed from a CUDA graph; "
                   "hbm_frac uses the measured copy bandwidth; 'gathered' and 'unfused' take "
                   "full-width (d_k = 128) q/k and keep 64 channels per head")
    res["launches"] = launches
    return res


def bench_prologue(args, torch, binding, d, idx, dp, o, peaks, barrier, max_over_ranks, world):
    """The pruning prologue on the prefill workload's full-width bf16 q and k
    (d_k = 128 -> 64 kept channels per head): the prologue alone (two
    launches), and prologue + d_k' = 64 prefill as one pruned pipeline.
    Prologue bytes per row: the full-width row read (a random half of the
    channels touches every 32-byte sector) plus the kept row written."""
    B, T, H, Kin = d["q"].shape
    Kout = idx.shape[-1]
    V = o.shape[-1]
    rows = B * T * H
    qg = torch.empty((B, T, H, Kout), dtype=torch.bfloat16, device="cuda")
    kg = torch.empty_like(qg)
    ST = torch.empty((B, H, V, Kout), dtype=torch.float32, device="cuda")

    def pro():
        binding.gdn_gather_normalize(d["q"], idx, qg, B * T, H, Kin, Kout, binding.GDN_BF16)
        binding.gdn_gather_normalize(d["k"], idx, kg, B * T, H, Kin, Kout, binding.GDN_BF16)

    wsb = binding.gdn_prefill_two_pass_workspace_size(B, T, H, Kout, V, binding.GDN_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def pipeline():
        pro()
        binding.gdn_prefill(qg, kg, dp["v"], dp["alpha"], dp["beta"], None, o, ST, B, T, H,
                            Kout, V, binding.GDN_BF16, ws, wsb)

    # the prologue inside the prefill's key-side pass (no separate pass)
    wsg = binding.gdn_prefill_gathered_workspace_size(B, T, H, Kin, Kout, V, binding.GDN_BF16)
    wg = torch.empty(wsg, dtype=torch.uint8, device="cuda")

    def gathered():
        binding.gdn_prefill_gathered(d["q"], d["k"], idx, Kin, dp["v"], dp["alpha"], dp["beta"],
                                     None, o, ST, B, T, H, Kout, V, binding.GDN_BF16, wg, wsg)

    tp, _ = time_calls(pro, args.steps, args.warmup, torch, barrier)
    tp = max_over_ranks(tp)
    tl, _ = time_calls(pipeline, args.steps, args.warmup, torch, barrier)
    tl = max_over_ranks(tl)
    tg, _ = time_calls(gathered, args.steps, args.warmup, torch, barrier)
    tg = max_over_ranks(tg)
    byts = 2 * rows * (2 * Kin + 2 * Kout)
    gbs = byts / (tp / args.steps / 1e3) / 1e9
    return {"workload": f"B={B} T={T} H={H} bf16 q and k, d_k {Kin} -> {Kout}",
            "prologue_us": tp / args.steps * 1e3, "prologue_gbs": gbs,
            "prologue_hbm_frac": gbs / peaks["hbm_gbs"],
            "pipeline_ms_per_step": tl / args.steps,
            "pipeline_tokens_per_s": B * T * world * args.steps / (tl / 1e3),
            "gathered_ms_per_step": tg / args.steps,
            "gathered_tokens_per_s": B * T * world * args.steps / (tg / 1e3),
            "gathered_speedup_vs_pipeline": tl / tg,
            "gathered_api": "gdn_prefill_gathered (prologue inside the key-side pass)",
            "launches": args.steps * (6 + 2)}


def bench_truncation(args, torch, binding, d, ST, barrier, max_over_ranks, world):
    """Rank-r truncation ("How much of a Gated DeltaNet state is used" blog,
    Sec. 3): one gdn_state_truncate call on the 128 final states of the
    headline run (r = 32; the kernel also returns every singular value), and
    the headline prefill run in 256-token segments with the carried state cut
    to rank 32 at each of the 15 boundaries."""
    B, T, H, K = d["k"].shape
    V = d["v"].shape[-1]
    S = ST.clone()
    sig = torch.empty((B * H, min(V, K)), device="cuda")

    def trunc():
        S.copy_(ST)
        binding.gdn_state_truncate(S, B * H, V, K, 32, sig, 30)

    steps = max(3, min(args.steps, 10))
    tt, _ = time_calls(trunc, steps, 2, torch, barrier)
    status = binding.gdn_get_last_device_status()
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    S_T = torch.empty_like(ST)

    def seg():
        binding.gdn_prefill_truncated(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o,
                                      S_T, B, T, H, K, V, binding.GDN_BF16, 256, 32, 30)

    ts, _ = time_calls(seg, steps, 2, torch, barrier)
    ts = max_over_ranks(ts)
    return {"state_truncate_ms": max_over_ranks(tt) / steps, "states": B * H, "r": 32,
            "includes": "a 8 MB state copy per call (the truncation works in place)",
            "device_status": status,
            "segmented_prefill": {"seg_len": 256, "r": 32, "ms_per_step": ts / steps,
                                  "tokens_per_s": B * T * world / (ts / steps / 1e3)},
            "sigma1_median": float(sig[:, 0].median().item())}


def bench_drrqr(args, torch, binding, inputs, peaks, barrier, max_over_ranks):
    """DRRQR channel selection on calibration activations of the prefill
    workload's size (B=8, T=4096, H=16, d_k=128, bf16): the Gram on the
    tensor cores (HBM-bound: every calibration byte read once) and the
    per-head selection of 64 channels with f = 2."""
    k, q = inputs.make_calibration()
    B, T, H, K = k.shape
    dk, dq = to_dev_bf16(k, torch), to_dev_bf16(q, torch)
    del k, q
    G = torch.empty((H, K, K), device="cuda")
    need = binding.gdn_channel_gram_workspace_size(B, T, H, K)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def gram():
        binding.gdn_channel_gram(dk, dq, B, T, H, K, binding.GDN_BF16, G, ws, need)

    steps = max(3, min(args.steps, 10))
    tg, per = time_calls(gram, steps, 3, torch, barrier)
    tg = max_over_ranks(tg)
    byts = 2 * B * T * H * K * 2
    gbs = byts / (statistics.mean(per) / 1e3) / 1e9
    idx = torch.empty((H, 64), dtype=torch.int32, device="cuda")
    rho = torch.empty(H, device="cuda")
    sw = torch.empty(H, dtype=torch.int32, device="cuda")

    def select():
        binding.gdn_drrqr_select(G, H, K, 64, 2.0, 1000, idx, rho, sw)

    ts, _ = time_calls(select, 3, 1, torch, barrier)
    return {"workload": "calibration k, q: B=8 T=4096 H=16 d_k=128 bf16 -> 64 channels, f=2",
            "gram_ms": tg / steps, "gram_gbs": gbs, "gram_hbm_frac": gbs / peaks["hbm_gbs"],
            "select_ms": max_over_ranks(ts) / 3, "swaps_per_head": sw.cpu().tolist(),
            "rho_max": float(rho.max().item())}


def bench_fp32(args, torch, binding, inputs, peaks, barrier, max_over_ranks, world):
    """All-fp32 mode: gdn_prefill with float32 q, k, v, o on the prefill
    workload's shapes, and the tiny 32 x 32 workload (B=1, H=1, T=256)."""
    out = {}
    for name, p in (("prefill_shapes", inputs.make_prefill(dtype="fp32")),
                    ("tiny_32x32", inputs.make_tiny())):
        B, T, H, K = p.k.shape
        V = p.v.shape[-1]
        f = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()  # noqa: E731
        q, k, v, al, be = f(p.q), f(p.k), f(p.v), f(p.alpha), f(p.beta)
        o = torch.empty((B, T, H, V), device="cuda")
        ST = torch.empty((B, H, V, K), device="cuda")

        def step():
            binding.gdn_prefill(q, k, v, al, be, None, o, ST, B, T, H, K, V, binding.GDN_FP32)

        steps = max(3, min(args.steps, 10))
        tot, _ = time_calls(step, steps, 2, torch, barrier)
        ms = max_over_ranks(tot) / steps
        byts = B * T * H * (4 * 2 * K + 4 * 2 * V + 8) + 4 * B * H * V * K
        out[name] = {"shape": f"B={B} T={T} H={H} d_k={K} d_v={V}", "ms_per_step": ms,
                     "tokens_per_s": B * T * world / (ms / 1e3),
                     "achieved_gbs": byts / (ms / 1e3) / 1e9}
    out["note"] = "token-by-token CUDA-core kernel (scalar gate); float32 q/k/v/o"
    return out


def gated_bytes(B, T, H, K, V, gate):
    """Algorithmic HBM bytes of a gated prefill: bf16 q, k, v, o; float32
    per-channel alpha; beta (KDA) or b and w (GDN2); S_T."""
    per = 2 * 2 * K + 2 * 2 * V + 4 * K + (4 if gate == "kda" else 4 * K + 4 * V)
    return B * T * H * per + 4 * B * H * V * K


def bench_gated(args, torch, binding, inputs, peaks, barrier, max_over_ranks, world):
    """KDA and GDN2 prefill on the prefill workload's shapes (B=8, T=4096,
    H=16, d_k=d_v=128, bf16): the chunkwise tensor-core form
    (gdn_prefill_gated_chunked, key-side pass + state pass) and the
    token-by-token kernel (gdn_prefill_gated)."""
    out = {}
    for gate in ("kda", "gdn2"):
        p = inputs.make_channel_gated(gate=gate, T=args.gated_tokens)
        B, T, H, K = p.k.shape
        V = p.v.shape[-1]
        dq, dk, dv = to_dev_bf16(p.q, torch), to_dev_bf16(p.k, torch), to_dev_bf16(p.v, torch)
        f32 = lambda x: None if x is None else torch.from_numpy(x).cuda()  # noqa: E731
        al, be, bg, wg = f32(p.alpha), f32(p.beta), f32(p.b), f32(p.w)
        del p
        o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
        ST = torch.empty((B, H, V, K), dtype=torch.float32, device="cuda")
        code = binding.GATES[gate]
        need = binding.gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, code,
                                                                binding.GDN_BF16)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")

        def chunked():
            binding.gdn_prefill_gated_chunked(dq, dk, dv, al, be, bg, wg, None, o, ST, B, T, H,
                                              K, V, code, binding.GDN_BF16, ws, need)

        def token():
            binding.gdn_prefill_gated(dq, dk, dv, al, be, bg, wg, None, o, ST, B, T, H, K, V,
                                      code, binding.GDN_BF16)

        steps = max(3, min(args.steps, 10))
        tc, _ = time_calls(chunked, steps, 3, torch, barrier)
        mc = max_over_ranks(tc) / steps
        status = binding.gdn_get_last_device_status()
        tt, _ = time_calls(token, 3, 1, torch, barrier)
        mt = max_over_ranks(tt) / 3
        byts = gated_bytes(B, T, H, K, V, gate)
        gbs = byts / (mc / 1e3) / 1e9
        out[gate] = {"ms_per_step": mc, "tokens_per_s": B * T * world / (mc / 1e3),
                     "achieved_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                     "algorithmic_bytes": byts,
                     # key-side and state passes; GDN2 adds its write-content kernel
                     "launches": (3 if gate == "gdn2" else 2) * steps,
                     "workspace_bytes": need, "device_status": status,
                     "token_kernel": {"ms_per_step": mt,
                                      "tokens_per_s": B * T * world / (mt / 1e3),
                                      "hbm_frac": byts / (mt / 1e3) / 1e9 / peaks["hbm_gbs"]},
                     "chunked_speedup": mt / mc}
        del dq, dk, dv, al, be, bg, wg, o, ST, ws
    out["workload"] = (f"B=8 T={args.gated_tokens} H=16 d_k=d_v=128 bf16, per-channel decay")
    out["api"] = ("gdn_prefill_gated_chunked (key-side pass over all chunks + state pass); "
                  "token_kernel: gdn_prefill_gated")
    out["note"] = ("bytes = q, k, v, o, gates, S_T (the algorithmic minimum); the chunked form "
                   "also moves its 64.5 KiB (KDA) / 80.5 KiB (GDN2) per chunk of key-side "
                   "operands through HBM")
    return out


def bench_long(args, torch, binding, inputs, peaks, barrier, max_over_ranks, world):
    """Long-context prefill (B=1, T=65536, H=16, d_k=d_v=128, alpha in
    [0.9995, 0.9999], keys in a narrow cone) and the stable rank of its final
    states.  Few heads and a long sequence: the prefill runs segment-parallel,
    in the two-pass form (workspace of gdn_prefill_two_pass_workspace_size)."""
    p = inputs.make_long()
    B, T, H, K = p.k.shape
    V = p.v.shape[-1]
    d = problem_to_dev(p, torch)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, V, K), dtype=torch.float32, device="cuda")
    wsb = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    wsb1 = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")

    def step():
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, ws, wsb)

    def step1():  # one-pass form: the segment scratch only
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, ws, wsb1)

    steps = max(3, min(args.steps, 10))
    tot1, _ = time_calls(step1, steps, 3, torch, barrier)
    tot1 = max_over_ranks(tot1)
    tot, per = time_calls(step, steps, 3, torch, barrier)
    tot = max_over_ranks(tot)
    ms = tot / steps
    f2 = torch.empty(B * H, device="cuda")
    s1 = torch.empty_like(f2)
    er = torch.empty_like(f2)
    binding.gdn_state_rank(ST, B * H, V, K, f2, s1, er, 2000, 0.0)
    return {"workload": "B=1 T=65536 H=16 d_k=d_v=128 bf16, alpha U[0.9995,0.9999], cone keys",
            "ms_per_step": ms, "tokens_per_s": B * T * world / (ms / 1e3),
            "achieved_gbs": prefill_bytes(B, T, H, K, V) / (ms / 1e3) / 1e9,
            "hbm_frac": prefill_bytes(B, T, H, K, V) / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "workspace_bytes": wsb,
            "one_pass_ms_per_step": tot1 / steps,
            "stable_rank_per_head": [round(float(x), 3) for x in er.cpu()]}


def bench_e2e(p, torch, binding, args, barrier, max_over_ranks, world, window=512):
    """The same prefill through the C ABI on pinned HOST buffers
    (gdn_prefill_host): every step copies its inputs host->device and o and
    S_T device->host, pipelined with the recurrence over 512-token windows;
    all of it inside the timed region."""
    B, T, H, K = p.k.shape
    V = p.v.shape[-1]
    from gated_delta_rule_49_gb300 import inputs
    hq = torch.from_numpy(inputs.bf16_bits(p.q).view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(inputs.bf16_bits(p.k).view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(inputs.bf16_bits(p.v).view(np.int16)).view(torch.bfloat16).pin_memory()
    ha = torch.from_numpy(np.ascontiguousarray(p.alpha)).pin_memory()
    hb = torch.from_numpy(np.ascontiguousarray(p.beta)).pin_memory()
    ho = torch.empty((B, T, H, V), dtype=torch.bfloat16).pin_memory()
    hS = torch.empty((B, H, V, K), dtype=torch.float32).pin_memory()
    need = binding.gdn_prefill_host_workspace_size(B, T, H, K, V, binding.GDN_BF16, window)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def step():
        binding.gdn_prefill_host(hq, hk, hv, ha, hb, None, ho, hS, B, T, H, K, V,
                                 binding.GDN_BF16, window, ws, need)

    steps = max(3, min(args.steps, 10))
    tot, _ = time_calls(step, steps, 2, torch, barrier)
    tot = max_over_ranks(tot)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, ha, hb))
    d2h = ho.numel() * ho.element_size() + hS.numel() * hS.element_size()
    return {"value": B * T * world * steps / (tot / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": f"gdn_prefill_host, pinned host buffers, {window}-token windows",
            "copy_gbs": (h2d + d2h) / (tot / steps / 1e3) / 1e9}


# ----------------------------------------------------------------- oracle arm
def oracle_sample(p, seqs):
    """`seqs` distinct (b, h) sequences of the workload, evenly spread, full length."""
    B, T, H, K = p.k.shape
    seqs = min(seqs, B * H)
    if seqs == B * H:
        return p
    step = (B * H) // seqs
    pick = [((j * step) // H, (j * step) % H) for j in range(seqs)]
    from gated_delta_rule_49_gb300 import inputs
    subs = [inputs.take_sequences(p, [b], [h]) for b, h in pick]
    cat = lambda xs: np.concatenate(xs, axis=0)  # noqa: E731
    return inputs.Problem(p.name, p.dtype, cat([s.q for s in subs]), cat([s.k for s in subs]),
                          cat([s.v for s in subs]), cat([s.alpha for s in subs]),
                          cat([s.beta for s in subs]), None, {})


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(p, seqs=None, reps=1, single_seqs=2):
    """The float64 oracle on the host cores: the whole workload on every core
    (one thread per independent sequence), and a few whole sequences on one
    thread."""
    import oracle
    cores = os.cpu_count() or 1
    B, T, H, K = p.k.shape
    seqs = seqs or B * H  # the whole workload: ~1 s on 16 cores
    sub = oracle_sample(p, seqs)
    threads = min(cores, seqs)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.recurrence(sub.q, sub.k, sub.v, sub.alpha, sub.beta, threads=threads)
    dt = (time.perf_counter() - t0) / reps
    token_heads = seqs * T
    one = oracle_sample(p, single_seqs)
    t0 = time.perf_counter()
    oracle.recurrence(one.q, one.k, one.v, one.alpha, one.beta, threads=1)
    dt1 = time.perf_counter() - t0
    return {"value": token_heads / H / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "nproc": cores, "cpu_model": cpu_model(),
            "single_thread": {"value": single_seqs * T / H / dt1, "unit": "tokens/s",
                              "wall_s": dt1,
                              "sample": f"{single_seqs} (b, h) sequences x {T} tokens, one thread"},
            "sample": f"{seqs} of {B * H} (b, h) sequences x {T} tokens, float64 C oracle; "
                      f"tokens/s = sequences*T/H / wall time ({dt:.2f} s)"}


def headline_config(W, world):
    """The `config` object both arms print for the headline workload."""
    return dict(W, l2="inputs larger than L2 (537 MB per step)",
                parallelism=f"independent batch per GPU x{world}")


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample of the
    headline workload (whole sequences) on the host cores."""
    if rank != 0:
        return None
    from gated_delta_rule_49_gb300 import inputs
    import oracle
    oracle.build()
    W = WORKLOAD
    Bw = args.ref_batch or W["B"]
    p = inputs.make_prefill(B=Bw, T=W["T"], H=W["H"], K=W["d_k"], V=W["d_v"])
    cores = os.cpu_count() or 1
    seqs = min(cores, 16)
    sub = oracle_sample(p, seqs)
    T, H = W["T"], W["H"]
    for _ in range(args.warmup):
        oracle.recurrence(sub.q[:, :256], sub.k[:, :256], sub.v[:, :256], sub.alpha[:, :256],
                          sub.beta[:, :256], threads=seqs)
    t0 = time.perf_counter()
    Tc = args.ref_tokens
    for _ in range(args.steps):
        oracle.recurrence(sub.q[:, :Tc], sub.k[:, :Tc], sub.v[:, :Tc], sub.alpha[:, :Tc],
                          sub.beta[:, :Tc], threads=seqs)
    dt = time.perf_counter() - t0
    value = seqs * Tc * args.steps / H / dt
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(dict(WORKLOAD, B=Bw), world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": seqs, "kind": "oracle",
                         "nproc": cores, "cpu_model": cpu_model(),
                         "sample": f"{seqs} (b, h) sequences x first {Tc} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------- main
def rank_sync(world, backend, device):
    """(barrier, max_over_ranks) for `world` ranks.  The path shards whole
    sequences across GPUs with no exchange step, so the only collectives are
    the timing barrier and the max over ranks of the elapsed time."""
    if world <= 1:
        return None, (lambda x: x)
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        if backend == "nccl":
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)

    def max_over_ranks(x):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return dist.barrier, max_over_ranks


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline prefill only")
    ap.add_argument("--only", default=None,
                    choices=["pruned", "prologue", "state_rank", "truncation", "drrqr",
                             "long_context", "gated", "fp32", "decode"],
                    help="headline prefill plus this one section (e.g. for a profiler run)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gated-tokens", type=int, default=4096,
                    help="T of the gated section's workload (a smaller case for profiling)")
    ap.add_argument("--cpu-seqs", type=int, default=None)
    ap.add_argument("--decode-reps", type=int, default=20)
    ap.add_argument("--ref-tokens", type=int, default=4096)
    ap.add_argument("--ref-batch", type=int, default=None,
                    help="batch of the workload the reference arm samples (default: the "
                         "headline batch); the sample is whole sequences either way")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        return

    import torch
    torch.cuda.set_device(local)
    barrier, max_over_ranks = rank_sync(world, "nccl", torch.device("cuda", local))

    line = run_ours(args, rank, world, barrier, max_over_ranks)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
