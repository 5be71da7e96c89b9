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


def expert_getter(w: wl.Workload, seed=0, cache: bool = True):
    """float64 weights of routed expert e for the oracle: the bf16 bits
    widened, or for FP8 workloads the oracle's own dequantisation of the codes.
    cache=False draws an expert again on every call (the oracle's forward
    asks for each expert once; the DeepSeek-sized experts would hold ~60 GB
    of float64 if all were kept)."""
    if w.weight_dtype != "e4m3":
        if cache:
            return wl.expert_getter_f64(w, seed)
        return lambda e: wl.expert_getter_f64(w, seed)(e)
    store = {}

    def get(e):
        if e in store:
            return store[e]
        q1, s1, b1, q2, s2, b2 = wl.gen_expert_e4m3(w, seed, e)
        v = (O.dequantize_rows(q1, s1), None if b1 is None else wl.bf16_bits_to_f64(b1),
             O.dequantize_rows(q2, s2), None if b2 is None else wl.bf16_bits_to_f64(b2))
        if cache:
            store[e] = v
        return v
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
                     w.aux_alpha, expert_getter(w, seed, cache=tokens is None),
                     shared_weights(w, seed),
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


# Row tiles of the expert GEMMs start at each expert's first row and are 128
# (single CTA) or 256 (CTA pair) rows high; every 256-row tile is two
# 128-row blocks, so covering the 128-row blocks covers both.
TILE_ROWS = 128


def tile_rows(offsets: np.ndarray, block: int = TILE_ROWS) -> np.ndarray:
    """The first and the last row of every `block`-row tile of every
    expert's row segment (the last tile of a segment is usually ragged)."""
    rows = []
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        for b in range(r0, r1, block):
            rows += [b, min(b + block, r1) - 1]
    return np.unique(np.array(rows, dtype=np.int64))


def tile_tokens(w: wl.Workload, x_bits, router, n_random: int = 48, seed: int = 123):
    """Tokens for a sampled full-size check: n_random random ones plus the
    tokens owning the first and the last row of every row tile of every
    expert, under the oracle's own routing and dispatch (so that every M-tile
    of the expert GEMMs, ragged last ones included, has an output row the
    oracle evaluates).  Returns (tokens, oracle offsets, oracle perm)."""
    Wg, bg, sel = router
    x = wl.bf16_bits_to_f64(x_bits)
    C = O.capacity(w.T, w.N, w.capacity_factor, w.min_capacity)
    if w.routing == "expert":
        d = O.expert_choice(O.gate_logits(x, Wg, bg), min(C, w.T))
        slots = w.N
    else:
        r = O.route(x, Wg, bg, sel, w.k)
        d = O.permute(r["idx"], w.N, C, w.drop_order)
        slots = w.k
    rows = tile_rows(d["offsets"])
    toks = set((d["perm"][rows] // slots).tolist())
    toks.update(sample_tokens(w.T, n_random, seed).tolist())
    return np.array(sorted(toks), dtype=np.int64), d["offsets"], d["perm"]


def assert_tiles_covered(offsets: np.ndarray, perm: np.ndarray, slots: int, checked) -> int:
    """Every TILE_ROWS-row tile of every expert segment holds at least one row
    whose token's output was compared.  Returns the number of tiles."""
    checked = set(np.asarray(checked).tolist())
    n = 0
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        for b in range(r0, r1, TILE_ROWS):
            toks = perm[b:min(b + TILE_ROWS, r1)] // slots
            assert checked.intersection(toks.tolist()), f"expert {e}: tile at row {b} unchecked"
            n += 1
    return n


def laux_close(gpu: float, ref: float):
    assert abs(gpu - ref) <= LAUX_RTOL * abs(ref) + 1e-12, (gpu, ref)


def math_ok(x):
    return math.isfinite(x)
