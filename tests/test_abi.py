"""The C ABI library loads, exports what include/gdn.h declares, and rejects
bad arguments on the host before any launch (no GPU needed: every call here
fails validation, so nothing touches a device)."""
import ctypes
import os
import re
import subprocess

import pytest

from gated_delta_rule_49_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing but the C ABI is exported
    assert {s for s in exported if not s.startswith("gdn_")} <= {"_init", "_fini"}


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 1, 2, 3):
        s = binding.status_string(code)
        assert s and s != "unknown status"
    assert binding.status_string(12345) == "unknown status"
    assert binding.gdn_version() >= 100


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation


def _prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, beta=FAKE, S0=None, o=FAKE, ST=FAKE, B=1, T=4,
             H=1, K=128, V=128, dt=0, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.gdn_prefill(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"], a["o"],
                           a["ST"], a["B"], a["T"], a["H"], a["K"], a["V"], a["dt"], a["ws"],
                           a["wsb"], a["stream"])


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, K=96) == binding.GDN_ERR_UNSUPPORTED
    assert _prefill(lib, K=128, V=64) == binding.GDN_ERR_UNSUPPORTED
    assert _prefill(lib, K=32, V=128) == binding.GDN_ERR_UNSUPPORTED
    assert _prefill(lib, B=-1) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, T=-3) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, dt=7) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, q=None) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, alpha=None) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, o=None, ST=None) == binding.GDN_ERR_INVALID_ARG
    assert _prefill(lib, k=FAKE + 8) == binding.GDN_ERR_ALIGNMENT
    assert _prefill(lib, S0=FAKE + 4) == binding.GDN_ERR_ALIGNMENT
    assert _prefill(lib, ST=FAKE + 2) == binding.GDN_ERR_ALIGNMENT
    # empty batch or head count: nothing to do, nothing launched
    assert _prefill(lib, B=0) == binding.GDN_OK
    assert _prefill(lib, H=0) == binding.GDN_OK


def test_decode_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, beta=FAKE, S=FAKE, o=FAKE, B=1, H=1, K=128,
                 V=128, dt=0)
        a.update(kw)
        return lib.gdn_decode_step(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S"],
                                   a["o"], a["B"], a["H"], a["K"], a["V"], a["dt"], None)
    assert call(K=16) == binding.GDN_ERR_UNSUPPORTED
    assert call(S=None) == binding.GDN_ERR_INVALID_ARG
    assert call(o=None) == binding.GDN_ERR_INVALID_ARG
    assert call(H=-1) == binding.GDN_ERR_INVALID_ARG
    assert call(dt=2) == binding.GDN_ERR_INVALID_ARG
    assert call(v=FAKE + 2) == binding.GDN_ERR_ALIGNMENT
    assert call(B=0) == binding.GDN_OK


def test_state_rank_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(S=FAKE, BH=1, V=128, K=128, f=FAKE, s=FAKE, e=FAKE, it=10, tol=1e-6)
        a.update(kw)
        return lib.gdn_state_rank(a["S"], a["BH"], a["V"], a["K"], a["f"], a["s"], a["e"],
                                  a["it"], ctypes.c_float(a["tol"]), None)
    assert call(V=129) == binding.GDN_ERR_INVALID_ARG
    assert call(K=0) == binding.GDN_ERR_INVALID_ARG
    assert call(it=0) == binding.GDN_ERR_INVALID_ARG
    assert call(tol=-1.0) == binding.GDN_ERR_INVALID_ARG
    assert call(tol=float("nan")) == binding.GDN_ERR_INVALID_ARG
    assert call(e=None) == binding.GDN_ERR_INVALID_ARG
    assert call(S=FAKE + 4) == binding.GDN_ERR_ALIGNMENT
    assert call(BH=0) == binding.GDN_OK


def test_workspace_query(lib):
    for K, V in ((32, 32), (64, 128), (128, 128)):
        assert binding.gdn_prefill_workspace_size(8, 4096, 16, K, V, 0) >= 0


def test_two_pass_workspace_query(lib):
    two = binding.gdn_prefill_two_pass_workspace_size
    # 128 sequences run one CTA each (no segment scratch): 16 KiB per 64-token chunk
    assert two(8, 4096, 16, 128, 128, binding.GDN_BF16) == 8 * 16 * 64 * 16384
    assert two(8, 4096, 16, 64, 128, binding.GDN_BF16) == 8 * 16 * 64 * 16384
    assert two(2, 65, 3, 128, 128, binding.GDN_BF16) == 2 * 3 * 2 * 16384  # ragged: 2 chunks
    for K, V in ((128, 128), (64, 128)):
        need = binding.gdn_prefill_workspace_size(1, 65536, 16, K, V, binding.GDN_BF16)
        assert two(1, 65536, 16, K, V, binding.GDN_BF16) >= need + 16 * 1024 * 16384
    # no two-pass form: float32, the (32, 32) variant, empty or invalid problems
    assert two(8, 4096, 16, 128, 128, binding.GDN_FP32) == 0
    assert two(1, 256, 1, 32, 32, binding.GDN_BF16) == 0
    assert two(0, 4096, 16, 128, 128, binding.GDN_BF16) == 0
    assert two(8, 0, 16, 128, 128, binding.GDN_BF16) == 0
    assert two(8, 4096, 16, 96, 128, binding.GDN_BF16) == 0


def test_gathered_prefill_workspace_and_validation(lib):
    size = binding.gdn_prefill_gathered_workspace_size
    bf = binding.GDN_BF16
    # key-side operands (16 KiB per chunk), then q' and k' (bf16, 64 channels)
    tok = 8 * 4096 * 16 * 64 * 2
    assert size(8, 4096, 16, 128, 64, 128, bf) == 8 * 16 * 64 * 16384 + 2 * tok
    # only full width 128 -> 64 kept channels at V = 128, bf16
    for args in ((8, 4096, 16, 96, 64, 128, bf), (8, 4096, 16, 128, 32, 128, bf),
                 (8, 4096, 16, 128, 64, 64, bf), (8, 4096, 16, 128, 64, 128, binding.GDN_FP32),
                 (0, 4096, 16, 128, 64, 128, bf)):
        assert size(*args) == 0
    f = lib.gdn_prefill_gathered
    dummy = 0x10000  # never dereferenced: every check below returns before a launch
    common = (dummy, dummy, dummy, 128, dummy, dummy, dummy, None, dummy, dummy)
    # unsupported widths / dtype
    assert f(dummy, dummy, dummy, 96, dummy, dummy, dummy, None, dummy, dummy, 2, 64, 3, 64, 128,
             bf, None, 0, None) == binding.GDN_ERR_UNSUPPORTED
    assert f(*common, 2, 64, 3, 64, 128, binding.GDN_FP32, None, 0, None) == \
        binding.GDN_ERR_UNSUPPORTED
    # neither output
    assert f(dummy, dummy, dummy, 128, dummy, dummy, dummy, None, None, None, 2, 64, 3, 64, 128,
             bf, None, 0, None) == binding.GDN_ERR_INVALID_ARG
    # misaligned index pointer
    assert f(dummy, dummy, dummy + 4, 128, dummy, dummy, dummy, None, dummy, dummy, 2, 64, 3, 64,
             128, bf, None, 0, None) == binding.GDN_ERR_ALIGNMENT
    # missing or short workspace
    assert f(*common, 2, 64, 3, 64, 128, bf, None, 0, None) == binding.GDN_ERR_WORKSPACE
    need = size(2, 64, 3, 128, 64, 128, bf)
    assert f(*common, 2, 64, 3, 64, 128, bf, dummy, need - 16, None) == binding.GDN_ERR_WORKSPACE


def test_selftest_rejects_bad_limit(lib):
    assert lib.gdn_selftest_wait_timeout(0, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_wait_timeout(1 << 40, None) == binding.GDN_ERR_INVALID_ARG


def test_prologue_rejects_bad_arguments(lib):
    F = FAKE
    assert lib.gdn_gather_normalize(F, F, F, 10, 2, 128, 48, 0, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_gather_normalize(F, F, F, 10, 2, 32, 64, 0, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_gather_normalize(F, None, F, 10, 2, 128, 64, 0, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_gather_normalize(F + 4, F, F, 10, 2, 128, 64, 0, None) == binding.GDN_ERR_ALIGNMENT
    assert lib.gdn_gather_normalize(F, F, F, 0, 2, 128, 64, 0, None) == binding.GDN_OK

    def dec(**kw):
        a = dict(q=F, k=F, idx=F, kin=128, v=F, al=F, be=F, S=F, o=F, B=1, H=1, K=64, V=128, dt=0)
        a.update(kw)
        return lib.gdn_decode_step_gathered(a["q"], a["k"], a["idx"], a["kin"], a["v"], a["al"],
                                            a["be"], a["S"], a["o"], a["B"], a["H"], a["K"],
                                            a["V"], a["dt"], None)
    assert dec(kin=32) == binding.GDN_ERR_INVALID_ARG
    assert dec(K=48) == binding.GDN_ERR_UNSUPPORTED
    assert dec(idx=None) == binding.GDN_ERR_INVALID_ARG
    assert dec(idx=F + 4) == binding.GDN_ERR_ALIGNMENT
    assert dec(B=0) == binding.GDN_OK


def test_gated_rejects_bad_arguments(lib):
    F = FAKE

    def pre(**kw):
        a = dict(q=F, k=F, v=F, al=F, be=F, b=None, w=None, S0=None, o=F, ST=F, B=1, T=4, H=1,
                 K=128, V=128, gate=binding.GDN_GATE_KDA, dt=0)
        a.update(kw)
        return lib.gdn_prefill_gated(a["q"], a["k"], a["v"], a["al"], a["be"], a["b"], a["w"],
                                     a["S0"], a["o"], a["ST"], a["B"], a["T"], a["H"], a["K"],
                                     a["V"], a["gate"], a["dt"], None)
    assert pre(gate=3) == binding.GDN_ERR_INVALID_ARG
    assert pre(K=96) == binding.GDN_ERR_UNSUPPORTED
    assert pre(be=None) == binding.GDN_ERR_INVALID_ARG            # KDA needs beta
    assert pre(b=F, w=F) == binding.GDN_ERR_INVALID_ARG           # ... and no b / w
    assert pre(gate=binding.GDN_GATE_GDN2) == binding.GDN_ERR_INVALID_ARG  # GDN2: b, w, no beta
    assert pre(gate=binding.GDN_GATE_GDN2, be=None, b=F) == binding.GDN_ERR_INVALID_ARG
    assert pre(o=None, ST=None) == binding.GDN_ERR_INVALID_ARG
    assert pre(al=F + 4) == binding.GDN_ERR_ALIGNMENT
    assert pre(gate=binding.GDN_GATE_GDN2, be=None, b=F, w=F + 8) == binding.GDN_ERR_ALIGNMENT
    assert pre(B=0) == binding.GDN_OK

    def dec(**kw):
        a = dict(q=F, k=F, v=F, al=F, be=None, b=F, w=F, S=F, o=F, B=1, H=1, K=64, V=128,
                 gate=binding.GDN_GATE_GDN2, dt=0)
        a.update(kw)
        return lib.gdn_decode_step_gated(a["q"], a["k"], a["v"], a["al"], a["be"], a["b"],
                                         a["w"], a["S"], a["o"], a["B"], a["H"], a["K"], a["V"],
                                         a["gate"], a["dt"], None)
    assert dec(be=F) == binding.GDN_ERR_INVALID_ARG
    assert dec(w=None) == binding.GDN_ERR_INVALID_ARG
    assert dec(S=None) == binding.GDN_ERR_INVALID_ARG
    assert dec(K=16) == binding.GDN_ERR_UNSUPPORTED
    assert dec(dt=5) == binding.GDN_ERR_INVALID_ARG
    assert dec(b=F + 4) == binding.GDN_ERR_ALIGNMENT
    assert dec(B=0) == binding.GDN_OK


def test_truncation_rejects_bad_arguments(lib):
    F = FAKE
    assert lib.gdn_state_truncate(F, 2, 128, 128, 0, None, 30, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_state_truncate(F, 2, 128, 128, 4, None, 0, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_state_truncate(F, 2, 128, 96, 4, None, 30, None) == binding.GDN_ERR_UNSUPPORTED
    assert lib.gdn_state_truncate(F + 4, 2, 128, 128, 4, None, 30, None) == binding.GDN_ERR_ALIGNMENT
    assert lib.gdn_state_truncate(F, 2, 128, 128, 4, F + 8, 30, None) == binding.GDN_ERR_ALIGNMENT
    # nothing to cut and no singular values asked: returns before any launch
    assert lib.gdn_state_truncate(F, 2, 128, 128, 128, None, 30, None) == binding.GDN_OK
    assert lib.gdn_state_truncate(F, 0, 128, 128, 4, None, 30, None) == binding.GDN_OK

    def pre(**kw):
        a = dict(q=F, k=F, v=F, al=F, be=F, S0=None, o=F, ST=F, B=1, T=300, H=1, K=128, V=128,
                 dt=0, seg=256, r=8, sw=30)
        a.update(kw)
        return lib.gdn_prefill_truncated(a["q"], a["k"], a["v"], a["al"], a["be"], a["S0"],
                                         a["o"], a["ST"], a["B"], a["T"], a["H"], a["K"],
                                         a["V"], a["dt"], a["seg"], a["r"], a["sw"], None, 0,
                                         None)
    assert pre(ST=None) == binding.GDN_ERR_INVALID_ARG
    assert pre(seg=0) == binding.GDN_ERR_INVALID_ARG
    assert pre(r=0) == binding.GDN_ERR_INVALID_ARG
    assert pre(sw=1001) == binding.GDN_ERR_INVALID_ARG
    assert pre(K=32) == binding.GDN_ERR_UNSUPPORTED
    assert pre(be=None) == binding.GDN_ERR_INVALID_ARG
    assert pre(o=F + 2) == binding.GDN_ERR_ALIGNMENT
    assert pre(H=0) == binding.GDN_OK


def test_drrqr_rejects_bad_arguments(lib):
    F = FAKE
    ws = binding.gdn_channel_gram_workspace_size(8, 4096, 16, 128)
    assert ws > 0 and binding.gdn_channel_gram_workspace_size(8, 4096, 16, 64) == 0
    g = lambda **kw: lib.gdn_channel_gram(kw.get("k", F), kw.get("q", F), kw.get("B", 8),  # noqa: E731
                                          kw.get("T", 4096), kw.get("H", 16), kw.get("K", 128),
                                          kw.get("dt", 0), kw.get("G", F), kw.get("ws", F),
                                          kw.get("wsb", ws), None)
    assert g(K=64) == binding.GDN_ERR_UNSUPPORTED
    assert g(dt=1) == binding.GDN_ERR_UNSUPPORTED
    assert g(dt=4) == binding.GDN_ERR_INVALID_ARG
    assert g(G=None) == binding.GDN_ERR_INVALID_ARG
    assert g(k=F + 2) == binding.GDN_ERR_ALIGNMENT
    assert g(wsb=ws - 1) == binding.GDN_ERR_WORKSPACE
    assert g(ws=None) == binding.GDN_ERR_WORKSPACE
    assert g(H=0) == binding.GDN_OK

    def sel(**kw):
        a = dict(G=F, H=16, n=128, k=64, f=2.0, sw=100, idx=F)
        a.update(kw)
        return lib.gdn_drrqr_select(a["G"], a["H"], a["n"], a["k"], ctypes.c_float(a["f"]),
                                    a["sw"], a["idx"], None, None, None)
    assert sel(k=128) == binding.GDN_ERR_INVALID_ARG
    assert sel(k=0) == binding.GDN_ERR_INVALID_ARG
    assert sel(n=129) == binding.GDN_ERR_INVALID_ARG
    assert sel(f=0.5) == binding.GDN_ERR_INVALID_ARG
    assert sel(f=float("nan")) == binding.GDN_ERR_INVALID_ARG
    assert sel(sw=-1) == binding.GDN_ERR_INVALID_ARG
    assert sel(idx=None) == binding.GDN_ERR_INVALID_ARG
    assert sel(G=F + 4) == binding.GDN_ERR_ALIGNMENT
    assert sel(H=0) == binding.GDN_OK


def test_host_prefill_rejects_bad_arguments(lib):
    F = FAKE
    need = binding.gdn_prefill_host_workspace_size(8, 4096, 16, 128, 128, 0, 512)
    assert need > 0 and binding.gdn_prefill_host_workspace_size(8, 4096, 16, 96, 128, 0, 512) == 0

    def call(**kw):
        a = dict(q=F, k=F, v=F, al=F, be=F, S0=None, o=F, ST=F, B=8, T=4096, H=16, K=128, V=128,
                 dt=0, w=512, ws=F, wsb=need)
        a.update(kw)
        return lib.gdn_prefill_host(a["q"], a["k"], a["v"], a["al"], a["be"], a["S0"], a["o"],
                                    a["ST"], a["B"], a["T"], a["H"], a["K"], a["V"], a["dt"],
                                    a["w"], a["ws"], a["wsb"], None)
    assert call(w=0) == binding.GDN_ERR_INVALID_ARG
    assert call(K=96) == binding.GDN_ERR_UNSUPPORTED
    assert call(o=None, ST=None) == binding.GDN_ERR_INVALID_ARG
    assert call(be=None) == binding.GDN_ERR_INVALID_ARG
    assert call(wsb=need - 1) == binding.GDN_ERR_WORKSPACE
    assert call(ws=F + 8) == binding.GDN_ERR_ALIGNMENT
    assert call(B=0) == binding.GDN_OK


def test_bounds_check_variant_builds_and_exports():
    """The debug variant (-DGDN_BOUNDS_CHECK) compiles from the same sources and
    exports the same C ABI."""
    import ctypes
    from gated_delta_rule_49_gb300 import build
    path = build.build(bounds_check=True)
    dbg = ctypes.CDLL(path)
    for name in binding.EXPORTS:
        assert hasattr(dbg, name), name
