"""CPU tests of the C ABI library: it loads without a GPU, exports every symbol
include/moe.h declares, and rejects bad arguments on the host before any
device call (fake, never-dereferenced pointers)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_72_b300 import _lib
    return _lib.load()


def _declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from sparse_mixture_experts_72_b300 import _lib
    decl = _declared()
    assert decl, "no declarations parsed"
    for name in decl:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert sorted(_lib.EXPORTED) == decl


def test_exports_nothing_else():
    import subprocess
    from sparse_mixture_experts_72_b300 import _lib
    r = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                       text=True)
    if r.returncode != 0:
        pytest.skip("nm unavailable")
    syms = [ln.split()[-1] for ln in r.stdout.splitlines() if " T " in ln]
    ours = [s for s in syms if not s.startswith("_")]
    assert sorted(ours) == _declared(), ours


def _cfg(**kw):
    from sparse_mixture_experts_72_b300._lib import MoeConfig
    d = dict(T=64, H=32, F=128, N=4, k=2, capacity_factor=0.0, F_shared=0, aux_alpha=0.01)
    d.update(kw)
    return MoeConfig(**d)


def test_host_shape_functions(lib):
    from oracle import moe_oracle as O
    for T, N, cf in [(32768, 64, 1.25), (4096, 8, 2.0), (100, 8, 1.0), (777, 12, 1.25),
                     (64, 4, 0.0), (40, 16, 0.1), (0, 8, 1.0)]:
        c = _cfg(T=T, N=N, capacity_factor=cf, k=1)
        want = O.capacity(T, N, cf)
        assert lib.moe_capacity(C.byref(c)) == (-1 if want is None else want)
        R = T if want is None else min(T, want * N)
        assert lib.moe_max_rows(C.byref(c)) == R
    c = _cfg()
    assert lib.moe_workspace_size(C.byref(c)) > 0
    assert lib.moe_workspace_size(C.byref(_cfg(k=5))) == 0  # k > N is invalid
    assert lib.moe_workspace_size(None) == 0
    # min_capacity raises a smaller capacity, only when a factor is given
    for T, N, cf, mc in [(40, 16, 0.1, 4), (32768, 64, 1.25, 4), (64, 4, 1.0, 20), (64, 4, 0.0, 4)]:
        want = O.capacity(T, N, cf, mc)
        c = _cfg(T=T, N=N, capacity_factor=cf, k=1, min_capacity=mc)
        assert lib.moe_capacity(C.byref(c)) == (-1 if want is None else want)
    # expert choice: N * min(C, T) rows; needs a capacity factor
    c = _cfg(T=300, N=6, capacity_factor=1.5, k=1, routing=1)
    assert lib.moe_max_rows(C.byref(c)) == 6 * 75
    c = _cfg(T=64, N=4, capacity_factor=8.0, k=1, routing=1)
    assert lib.moe_max_rows(C.byref(c)) == 4 * 64
    assert lib.moe_workspace_size(C.byref(_cfg(routing=1, capacity_factor=0.0))) == 0
    for bad in (dict(routing=2), dict(activation=3), dict(drop_order=2), dict(min_capacity=-1),
                dict(weight_dtype=2)):
        assert lib.moe_workspace_size(C.byref(_cfg(**bad))) == 0, bad
    # E4M3 rows must start on 16-byte boundaries: H, F, F_shared multiples of 16
    assert lib.moe_workspace_size(C.byref(_cfg(weight_dtype=1))) > 0
    for bad in (dict(H=40), dict(F=136), dict(F_shared=72)):
        assert lib.moe_workspace_size(C.byref(_cfg(weight_dtype=1, **bad))) == 0, bad
        assert lib.moe_workspace_size(C.byref(_cfg(**bad))) > 0, bad


def _wcfg(w):
    from sparse_mixture_experts_72_b300 import _lib
    return _cfg(T=w.T, H=w.H, F=w.F, N=w.N, k=w.k, capacity_factor=w.capacity_factor,
                F_shared=w.F_shared, routing=_lib.ROUTING[w.routing],
                activation=_lib.ACTIVATION[w.activation], min_capacity=w.min_capacity,
                drop_order=_lib.DROP_ORDER[w.drop_order],
                weight_dtype=_lib.WEIGHT_DTYPE[w.weight_dtype])


def test_launch_names_cover_every_launch(lib):
    """One name per launch moe_forward enqueues; the expert FFN (shared
    expert included) runs as the operand-swapped decode launch exactly when
    the experts hold at most 64 rows on average, else as the token-row
    launch."""
    import moe_workloads as wl
    for w in list(wl.WORKLOADS.values()) + list(wl.TEST_WORKLOADS.values()):
        c = _wcfg(w)
        n = lib.moe_forward_num_launches(C.byref(c))
        names = [lib.moe_forward_launch_name(C.byref(c), i) for i in range(n + 1)]
        assert all(isinstance(x, bytes) for x in names[:n]) and names[n] is None, w.name
        names = [x.decode() for x in names[:n]]
        R = lib.moe_max_rows(C.byref(c))
        decode = R <= 64 * w.N
        assert ("expert_ffn_decode" in names) == (decode and (R > 0 or w.F_shared > 0)), w.name
        # the shared expert is a group of the expert-FFN launch on both paths
        assert "shared_ffn" not in names, w.name
        assert ("expert_ffn" in names) == (not decode and (R > 0 or w.F_shared > 0)), w.name
        assert names[-1] == "combine", w.name
    for name in ("mixtral_decode", "deepseek_decode", "mixtral_decode_fp8", "tiny"):
        c = _wcfg(wl.get_workload(name))
        n = lib.moe_forward_num_launches(C.byref(c))
        assert b"expert_ffn_decode" in [lib.moe_forward_launch_name(C.byref(c), i)
                                        for i in range(n)], name
    for name in ("moelayer", "mixtral_prefill", "deepseek_prefill", "switch_capacity"):
        c = _wcfg(wl.get_workload(name))
        n = lib.moe_forward_num_launches(C.byref(c))
        assert b"expert_ffn" in [lib.moe_forward_launch_name(C.byref(c), i)
                                 for i in range(n)], name
    assert lib.moe_forward_launch_name(C.byref(_cfg()), -1) is None


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every check fails before a device call


def _weights(**kw):
    from sparse_mixture_experts_72_b300._lib import MoeWeights
    d = dict(Wg=FAKE, bg=None, sel_bias=None, W1=FAKE, b1=None, W2=FAKE, b2=None, W1s=None,
             b1s=None, W2s=None, b2s=None, s1=None, s2=None, s1s=None, s2s=None)
    d.update(kw)
    return MoeWeights(**d)


def _forward(lib, cfg, weights, x=FAKE, out=FAKE, ws=FAKE * 16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.moe_workspace_size(C.byref(cfg)) or 1
    return lib.moe_forward(C.byref(cfg), C.byref(weights), x, out, None, ws, ws_bytes, None, None)


def test_rejects_bad_arguments_before_any_launch(lib):
    ok = _cfg()
    assert _forward(lib, _cfg(k=0), _weights()) == 1           # INVALID_ARG
    assert _forward(lib, _cfg(k=5), _weights()) == 1           # k > N
    assert _forward(lib, _cfg(T=-1), _weights()) == 1
    assert _forward(lib, _cfg(H=36), _weights()) == 2          # H % 8
    assert _forward(lib, _cfg(N=2000, k=2), _weights()) == 2   # N > MOE_MAX_EXPERTS
    assert _forward(lib, ok, _weights(Wg=None)) == 1           # required pointer
    assert _forward(lib, ok, _weights(W1=FAKE + 4)) == 2       # misaligned
    assert _forward(lib, ok, _weights(), x=FAKE + 2) == 2
    assert _forward(lib, _cfg(F_shared=64), _weights()) == 1   # shared weights missing
    assert _forward(lib, ok, _weights(), ws=None) == 3         # WORKSPACE
    assert _forward(lib, ok, _weights(), ws=FAKE * 16 + 16) == 3
    assert _forward(lib, ok, _weights(), ws_bytes=16) == 3
    # all checks pass: without a GPU the first device query fails cleanly
    # (never run with a GPU present: the fake pointers would reach a kernel)
    import torch
    if not torch.cuda.is_available():
        assert _forward(lib, ok, _weights()) == 6
    # E4M3 weights need their row scales (16-byte aligned); bf16 ignores them
    fp8 = _cfg(weight_dtype=1)
    assert _forward(lib, fp8, _weights()) == 1
    assert _forward(lib, fp8, _weights(s1=FAKE)) == 1
    assert _forward(lib, fp8, _weights(s1=FAKE, s2=FAKE + 4)) == 2
    assert _forward(lib, _cfg(weight_dtype=1, F_shared=64),
                    _weights(s1=FAKE, s2=FAKE, W1s=FAKE, W2s=FAKE)) == 1  # shared scales
    assert _forward(lib, _cfg(weight_dtype=1, H=40), _weights(s1=FAKE, s2=FAKE)) == 2
    if not torch.cuda.is_available():
        assert _forward(lib, fp8, _weights(s1=FAKE, s2=FAKE)) == 6
    assert lib.moe_status_string(3) == b"workspace missing, misaligned or too small"
    # widened entry points validate on the host as well
    ec = _cfg(routing=1, capacity_factor=1.0)
    assert lib.moe_expert_choice(C.byref(ok), FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None,
                                 None) == 1   # token-choice config
    assert lib.moe_expert_choice(C.byref(ec), FAKE + 4, None, FAKE, FAKE, FAKE, FAKE, None, None,
                                 None) == 2   # misaligned logits
    assert lib.moe_expert_choice(C.byref(ec), FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                 None) == 1   # l_aux without p_mean
    assert lib.moe_expert_choice(C.byref(_cfg(routing=1, capacity_factor=1.0, T=60000)), FAKE,
                                 None, FAKE, FAKE, FAKE, FAKE, None, None, None) == 2  # T too large
    assert lib.moe_update_sel_bias(C.byref(ok), None, FAKE, C.c_float(0.1), None) == 1
    assert lib.moe_permute(C.byref(ec), FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE * 16,
                           1 << 30, None) == 1   # expert choice has its own dispatch


def test_failure_injection_hook_validates_its_count(lib):
    # host-only: sets or clears a process-wide count, launches nothing
    assert lib.moe_debug_suppress_gemm_producer(-1) == 1   # INVALID_ARG
    assert lib.moe_debug_suppress_gemm_producer(3) == 0
    assert lib.moe_debug_suppress_gemm_producer(0) == 0
