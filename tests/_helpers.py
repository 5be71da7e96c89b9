"""Shared helpers for the GPU parity tests: upload seeded inputs, run the
oracle on the same bytes, and compare with the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import moe_workloads as wl
from oracle import moe_oracle as O

# Tolerances fixed by the target: probabilities 1e-5 absolute (fp32 router),
# L_aux 1e-5 relative, layer outputs |gpu - oracle| <= 1e-2 + 1e-2 |oracle|,
# near-tie margin 1e-5 in probability space.
PROB_ATOL = 1e-5
LAUX_RTOL = 1e-5
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
TIE_MARGIN = 1e-5


def bf16_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def f32_dev(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    """Device bf16 tensor -> float64 numpy (exact)."""
    return wl.bf16_bits_to_f64(t.detach().view(torch.int16).cpu().numpy().view(np.uint16))


def config_of(w: wl.Workload):
    import sparse_mixture_experts_72_b300 as m
    return m.MoEConfig(**w.config_kwargs())


def upload(w: wl.Workload, seed: int = 0, device="cuda"):
    """Seeded inputs on the device.  Returns (x_bits_host, weights, router_host)."""
    import sparse_mixture_experts_72_b300 as m
    d = wl.to_device(w, seed, device)
    weights = m.MoEWeights(**{k: d[k] for k in wl.WEIGHT_KEYS})
    return d["x_bits"], weights, wl.gen_router(w, seed)


def expert_getter(w: wl.Workload, seed=0):
    """float64 weights of routed expert e for the oracle: the bf16 bits
    widened, or for FP8 workloads the oracle's own dequantisation of the codes."""
    if w.weight_dtype != "e4m3":
        return wl.expert_getter_f64(w, seed)
    cache = {}

    def get(e):
        if e not in cache:
            q1, s1, b1, q2, s2, b2 = wl.gen_expert_e4m3(w, seed, e)
            cache[e] = (O.dequantize_rows(q1, s1), None if b1 is None else wl.bf16_bits_to_f64(b1),
                        O.dequantize_rows(q2, s2), None if b2 is None else wl.bf16_bits_to_f64(b2))
        return cache[e]
    return get


def shared_weights(w: wl.Workload, seed=0):
    if w.weight_dtype != "e4m3":
        return wl.shared_f64(w, seed)
    sh = wl.gen_shared_e4m3(w, seed)
    if sh is None:
        return None
    q1, s1, b1, q2, s2, b2 = sh
    return (O.dequantize_rows(q1, s1), None if b1 is None else wl.bf16_bits_to_f64(b1),
            O.dequantize_rows(q2, s2), None if b2 is None else wl.bf16_bits_to_f64(b2))


def oracle_forward(w: wl.Workload, x_bits, router, seed=0, tokens=None):
    Wg, bg, sel = router
    return O.forward(wl.bf16_bits_to_f64(x_bits), Wg, bg, sel, w.k, w.capacity_factor,
                     w.aux_alpha, expert_getter(w, seed), shared_weights(w, seed),
                     tokens=tokens, routing=w.routing, activation=w.activation,
                     min_capacity=w.min_capacity, drop_order=w.drop_order)


# A GPU choice that differs from the oracle's at a near tie must still be a
# top-k ranking of the oracle's float64 scores up to this logit slack (far
# below the 1e-5 probability margin that defines a near tie).
SCORE_SLACK = 1e-4


def check_routing(ref: dict, idx_gpu: np.ndarray, w_gpu: np.ndarray, k: int):
    """idx bit-exact except at near ties: tokens whose k-th/(k+1)-th
    selection-probability margin, or whose gap between adjacent chosen slots,
    is below TIE_MARGIN.  There the GPU's choice must still be a valid
    descending top-k of the oracle's scores.  Weights within PROB_ATOL
    elsewhere.  Returns the tokens whose choice differs (reported, not failed)."""
    idx_ref = ref["idx"]
    diff = np.nonzero((idx_gpu != idx_ref).any(axis=1))[0]
    near = np.minimum(ref["margin"], ref["order_margin"]) < TIE_MARGIN
    bad = [int(t) for t in diff if not near[t]]
    assert not bad, f"routing differs on {len(bad)} tokens that are not near ties, e.g. {bad[:5]}"
    s = ref["scores"]
    for t in diff:
        sg = s[t, idx_gpu[t]]
        assert len(set(idx_gpu[t].tolist())) == k, (t, idx_gpu[t])
        assert (np.diff(sg) <= SCORE_SLACK).all(), (t, idx_gpu[t], sg)
        rest = np.delete(s[t], idx_gpu[t])
        assert rest.size == 0 or sg.min() >= rest.max() - SCORE_SLACK, (t, idx_gpu[t])
    ok = np.setdiff1d(np.arange(idx_ref.shape[0]), diff)
    if ok.size:
        np.testing.assert_allclose(w_gpu[ok], ref["w"][ok], rtol=0, atol=PROB_ATOL)
    return [int(t) for t in diff]


def assert_close_out(gpu: np.ndarray, ref: np.ndarray, what="out"):
    err = np.abs(gpu - ref)
    lim = OUT_ATOL + OUT_RTOL * np.abs(ref)
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu {gpu[i]} oracle {ref[i]}")
    return float(err.max()) if err.size else 0.0


def sample_tokens(T: int, n: int, seed: int = 123) -> np.ndarray:
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    picks = set([0, T - 1, T // 2])
    picks.update(rng.choice(T, size=n - len(picks), replace=False).tolist())
    return np.array(sorted(picks)[:n])


def laux_close(gpu: float, ref: float):
    assert abs(gpu - ref) <= LAUX_RTOL * abs(ref) + 1e-12, (gpu, ref)


def math_ok(x):
    return math.isfinite(x)
