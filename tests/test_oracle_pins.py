"""Pins of the CPU oracle to things other than itself.

Each check compares the oracle with something the pages or the mathematics
fix: hand-worked fixtures under tests/golden (each with its source),
textbook values, closed forms, brute force on tiny inputs, library routines
(torch float64 softmax / topk / linear / gelu, numpy stable sort) and
invariants.  ``test_pins_catch_planted_mistakes`` plants plausible mistakes
in the oracle (on the CPU) and asserts that some pin fails for each.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

import moe_workloads as wl
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _logits_as_gate(L):
    """x = I_T, W_g = L^T so that the gate Linear reproduces the logits L exactly."""
    L = np.asarray(L, np.float64)
    T, N = L.shape
    return np.eye(T), L.T.copy()


# ---------------------------------------------------------------------------
# pin checks (plain functions so the planted-mistake test can rerun them)

def check_router_worked_example():
    g = _golden("router_worked_example.json")
    L = np.log(np.asarray([g["logits_exp"]], np.float64))
    x, Wg = _logits_as_gate(L)
    r = O.route(x, Wg, None, None, g["k"])
    np.testing.assert_allclose(r["probs"][0], g["probs"], rtol=0, atol=1e-15)
    assert r["idx"][0].tolist() == g["idx"]
    np.testing.assert_allclose(r["w"][0], g["w"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["margin"][0], g["margin"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["order_margin"][0], g["order_margin"], rtol=0, atol=1e-15)


def check_capacity_examples():
    for c in _golden("capacity_examples.json")["cases"]:
        assert O.capacity(c["T"], c["N"], c["cf"]) == c["C"], c


def check_permute_worked_example():
    g = _golden("permute_worked_example.json")
    idx = np.asarray(g["idx"])
    for key in ("capped", "unlimited"):
        case = g[key]
        C = O.capacity(g["T"], g["N"], case["cf"])
        if key == "capped":
            assert C == case["C"]
        d = O.permute(idx, g["N"], C)
        assert d["counts"].tolist() == g["counts"]
        for name in ("kept", "offsets", "perm", "inv"):
            assert d[name].tolist() == case[name], (key, name)
    P = np.full((g["T"], g["N"]), 1.0 / g["N"])
    lb = O.load_balance(P, np.asarray(g["counts"]), g["k"], 0.01)
    np.testing.assert_allclose(lb["f"], g["f"], rtol=0, atol=1e-15)


def check_laux_worked_examples():
    g = _golden("laux_worked_example.json")
    for c in g["cases"]:
        L = np.log(np.asarray(c["logits_exp"], np.float64))
        x, Wg = _logits_as_gate(L)
        r = O.route(x, Wg, None, None, c["k"])
        assert r["idx"].tolist() == c["idx"]
        d = O.permute(r["idx"], c["N"], None)
        lb = O.load_balance(r["probs"], d["counts"], c["k"], g["alpha"])
        np.testing.assert_allclose(lb["f"], c["f"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lb["p"], c["p"], rtol=0, atol=1e-15)
        assert abs(lb["l_aux"] - c["l_aux"]) <= 1e-15


def check_gelu_textbook():
    phi = _golden("gelu_textbook.json")["phi"]
    for z, p in phi.items():
        z = float(z)
        assert abs(O.gelu(np.array([z]))[0] - z * p) <= 1e-15 * max(1.0, abs(z)), z


def check_moelayer_worked_example():
    g = _golden("moelayer_worked_example.json")
    ex = [tuple(np.asarray(e[n], np.float64) for n in ("W1", "b1", "W2", "b2")) for e in g["experts"]]
    res = O.forward(np.asarray(g["x"]), np.asarray(g["Wg"]), np.asarray(g["bg"]), None,
                    g["k"], 0.0, 0.01, lambda e: ex[e])
    assert res["idx"].tolist() == g["idx"]
    np.testing.assert_allclose(res["out"], g["out"], rtol=1e-15, atol=1e-15)


def check_topk_bruteforce(seed=1):
    rng = np.random.default_rng(seed)
    for trial in range(200):
        N = int(rng.integers(1, 7))
        k = int(rng.integers(1, N + 1))
        T = int(rng.integers(1, 6))
        if trial % 2:
            s = rng.integers(-2, 3, size=(T, N)).astype(np.float64)   # many exact ties
        else:
            s = rng.standard_normal((T, N))
        idx = O.select_topk(s, k)[0]
        for t in range(T):
            # best subset: largest sum, then the lexicographically smallest index set
            best = max(itertools.combinations(range(N), k),
                       key=lambda c: (sum(s[t, i] for i in c), [-i for i in c]))
            # slot order: descending score, ties to the lower index
            want = sorted(best, key=lambda i: (-s[t, i], i))
            assert idx[t].tolist() == want, (s[t], k, idx[t], want)


def check_router_vs_torch(seed=2):
    rng = np.random.default_rng(seed)
    T, H, N, k = 50, 24, 10, 3
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((N, H)) / math.sqrt(H)
    bg = rng.standard_normal(N) * 0.3
    r = O.route(x, Wg, bg, None, k)
    logits = TF.linear(torch.from_numpy(x), torch.from_numpy(Wg), torch.from_numpy(bg))
    P = torch.softmax(logits, dim=-1)
    tw, ti = torch.topk(P, k, dim=-1)
    tw = tw / tw.sum(-1, keepdim=True)
    np.testing.assert_allclose(r["probs"], P.numpy(), rtol=1e-13, atol=1e-15)
    assert np.array_equal(r["idx"], ti.numpy())
    np.testing.assert_allclose(r["w"], tw.numpy(), rtol=1e-13, atol=1e-15)


def check_selection_bias(seed=3):
    """Selection follows l - b; weights stay the unbiased renormalised softmax."""
    rng = np.random.default_rng(seed)
    T, H, N, k = 40, 16, 8, 2
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((N, H)) / 4.0
    b = rng.uniform(-1.0, 1.0, N)
    r = O.route(x, Wg, None, b, k)
    logits = torch.from_numpy(x @ Wg.T)
    ti = torch.topk(logits - torch.from_numpy(b), k, dim=-1).indices
    assert np.array_equal(r["idx"], ti.numpy())
    P = torch.softmax(logits, -1)
    sel = torch.gather(P, 1, ti)
    np.testing.assert_allclose(r["w"], (sel / sel.sum(-1, keepdim=True)).numpy(), rtol=1e-13)
    # a large bias on expert 0 keeps it out of every selection
    b2 = np.zeros(N)
    b2[0] = 100.0
    assert not (O.route(x, Wg, None, b2, k)["idx"] == 0).any()


def check_zero_gate_all_ties():
    T, H, N, k = 7, 5, 6, 3
    r = O.route(np.ones((T, H)), np.zeros((N, H)), None, None, k)
    assert (r["idx"] == np.arange(k)[None, :]).all()
    np.testing.assert_allclose(r["w"], 1.0 / k, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["probs"], 1.0 / N, rtol=0, atol=1e-15)
    d = O.permute(r["idx"], N, None)
    assert abs(O.load_balance(r["probs"], d["counts"], k, 0.01)["l_aux"] - 0.01) < 1e-15


def check_weights_invariants(seed=4):
    rng = np.random.default_rng(seed)
    T, H, N, k = 200, 32, 16, 4
    r = O.route(rng.standard_normal((T, H)), rng.standard_normal((N, H)), None, None, k)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, rtol=0, atol=1e-12)
    assert (r["w"] >= 0).all()
    assert (np.diff(r["w"], axis=1) <= 0).all()
    assert (r["margin"] >= 0).all() and (r["order_margin"] >= 0).all()


def check_permute_vs_stable_sort(seed=5):
    rng = np.random.default_rng(seed)
    for trial in range(30):
        N = int(rng.integers(1, 20))
        k = int(rng.integers(1, min(N, 4) + 1))
        T = int(rng.integers(0, 300))
        # distinct experts per token, skewed toward low indices
        p = 1.0 / np.arange(1, N + 1) ** 1.1
        p /= p.sum()
        idx = np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)]) \
            if T else np.zeros((0, k), np.int64)
        cf = float(rng.choice([0.0, 0.5, 1.0, 1.25, 2.0]))
        C = O.capacity(T, N, cf)
        d = O.permute(idx, N, C)
        flat = idx.reshape(-1)
        # independent formulation: stable sort by expert, truncate each segment at C
        order = np.argsort(flat, kind="stable")
        counts = np.bincount(flat, minlength=N)
        assert np.array_equal(d["counts"], counts)
        kept_want = counts if C is None else np.minimum(counts, C)
        assert np.array_equal(d["kept"], kept_want)
        starts = np.concatenate([[0], np.cumsum(counts)])
        perm_want = np.concatenate([order[starts[e]:starts[e] + kept_want[e]] for e in range(N)]) \
            if N else np.zeros(0, np.int64)
        assert np.array_equal(d["perm"], perm_want)
        inv_want = np.full(flat.shape[0], -1)
        inv_want[perm_want] = np.arange(perm_want.shape[0])
        assert np.array_equal(d["inv"], inv_want)
        # invariants
        assert d["counts"].sum() == T * k
        assert d["offsets"][-1] == (d["inv"] >= 0).sum() == T * k - (d["inv"] < 0).sum()
        assert (np.diff(d["offsets"]) >= 0).all()
        for e in range(N):
            seg = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
            assert (np.diff(seg) > 0).all()
            assert (flat[seg] == e).all()


def _rand_layer(rng, T, H, F, N, with_bias=True):
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((N, H)) / math.sqrt(H)
    ex = []
    for _ in range(N):
        ex.append((rng.standard_normal((F, H)) / math.sqrt(H),
                   rng.standard_normal(F) * 0.1 if with_bias else None,
                   rng.standard_normal((H, F)) / math.sqrt(F),
                   rng.standard_normal(H) * 0.1 if with_bias else None))
    return x, Wg, ex


def _torch_ffn(x, W1, b1, W2, b2):
    t = lambda a: None if a is None else torch.from_numpy(np.asarray(a, np.float64))
    h = TF.gelu(TF.linear(t(x), t(W1), t(b1)), approximate="none")
    return TF.linear(h, t(W2), t(b2)).numpy()


def check_dense_reduction(seed=6):
    rng = np.random.default_rng(seed)
    for H, F in [(20, 48), (16, 16)]:   # the square case catches a transposed operand
        x, Wg, ex = _rand_layer(rng, 33, H, F, 1)
        res = O.forward(x, Wg, None, None, 1, 0.0, 0.01, lambda e: ex[e])
        np.testing.assert_allclose(res["out"], _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)


def check_identical_experts(seed=7):
    rng = np.random.default_rng(seed)
    x, Wg, ex = _rand_layer(rng, 40, 16, 24, 6)
    res = O.forward(x, Wg, rng.standard_normal(6), rng.uniform(-.1, .1, 6), 3, 0.0, 0.01,
                    lambda e: ex[0])
    np.testing.assert_allclose(res["out"], _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)


def check_shared_only(seed=8):
    rng = np.random.default_rng(seed)
    x, Wg, ex = _rand_layer(rng, 25, 16, 24, 4)
    zero = [(a, b, np.zeros_like(c), np.zeros_like(d)) for a, b, c, d in ex]
    sh = _rand_layer(rng, 1, 16, 40, 1)[2][0]
    res = O.forward(x, Wg, None, None, 2, 0.0, 0.01, lambda e: zero[e], shared=sh)
    np.testing.assert_allclose(res["out"], _torch_ffn(x, *sh), rtol=1e-12, atol=1e-12)


def check_linearity_in_w2(seed=9):
    rng = np.random.default_rng(seed)
    x, Wg, ex = _rand_layer(rng, 30, 12, 20, 5)
    dbl = [(a, b, 2 * c, 2 * d) for a, b, c, d in ex]
    o1 = O.forward(x, Wg, None, None, 2, 1.0, 0.01, lambda e: ex[e])["out"]
    o2 = O.forward(x, Wg, None, None, 2, 1.0, 0.01, lambda e: dbl[e])["out"]
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-12, atol=1e-13)


def check_expert_relabelling(seed=10):
    rng = np.random.default_rng(seed)
    N = 7
    x, Wg, ex = _rand_layer(rng, 35, 12, 20, N)
    bg = rng.standard_normal(N) * 0.2
    sb = rng.uniform(-.1, .1, N)
    pi = rng.permutation(N)
    o1 = O.forward(x, Wg, bg, sb, 3, 0.0, 0.01, lambda e: ex[e])
    o2 = O.forward(x, Wg[pi], bg[pi], sb[pi], 3, 0.0, 0.01, lambda e: ex[pi[e]])
    np.testing.assert_allclose(o2["out"], o1["out"], rtol=1e-12, atol=1e-13)
    assert abs(o2["l_aux"] - o1["l_aux"]) < 1e-14


def _moelayer_restated(x, Wg, bg, ex, k, cf=0.0, shared=None):
    """The pages' MoELayer loop ([SKILLS] §3.1: per slot, per expert, masked
    update) restated with torch float64 library routines, plus the capacity
    rule of [ARCH] §2.3 written as a cumulative count over assignments."""
    xt = torch.from_numpy(x)
    logits = TF.linear(xt, torch.from_numpy(Wg), None if bg is None else torch.from_numpy(bg))
    scores = torch.softmax(logits, dim=-1)
    ts, ti = torch.topk(scores, k, dim=-1)
    ts = ts / ts.sum(dim=-1, keepdim=True)
    T, N = scores.shape
    keep = torch.ones(T, k, dtype=torch.bool)
    if cf > 0:
        C = math.floor(T / N * cf)
        onehot = TF.one_hot(ti.reshape(-1), N)
        rank = (torch.cumsum(onehot, 0) - 1).gather(1, ti.reshape(-1, 1)).reshape(T, k)
        keep = rank < C
    out = torch.zeros_like(xt)
    for i in range(k):
        for e in range(N):
            mask = (ti[:, i] == e) & keep[:, i]
            if mask.any():
                y = _torch_ffn(x[mask.numpy()], *ex[e])
                out[mask] += ts[mask, i:i + 1] * torch.from_numpy(y)
    if shared is not None:
        out += torch.from_numpy(_torch_ffn(x, *shared))
    return out.numpy()


def check_moelayer_restatement(seed=11):
    rng = np.random.default_rng(seed)
    for (T, H, F, N, k, cf, sh) in [(64, 32, 128, 4, 2, 0.0, False), (90, 16, 24, 6, 2, 1.0, True),
                                    (120, 16, 24, 8, 1, 1.25, False)]:
        x, Wg, ex = _rand_layer(rng, T, H, F, N)
        bg = rng.standard_normal(N) * np.linspace(0, 1.5, N)
        shared = _rand_layer(rng, 1, H, 2 * F, 1)[2][0] if sh else None
        res = O.forward(x, Wg, bg, None, k, cf, 0.01, lambda e: ex[e], shared=shared)
        want = _moelayer_restated(x, Wg, bg, ex, k, cf, shared)
        np.testing.assert_allclose(res["out"], want, rtol=1e-12, atol=1e-12)


def check_tiny_workload_restatement():
    w = wl.WORKLOADS["tiny"]
    inp = wl.gen_all(w, 0)
    x = wl.bf16_bits_to_f64(inp["x"])
    get = wl.expert_getter_f64(w, 0)
    ex = [get(e) for e in range(w.N)]
    res = O.forward(x, inp["Wg"], inp["bg"], None, w.k, w.capacity_factor, w.aux_alpha, get)
    want = _moelayer_restated(x, inp["Wg"].astype(np.float64), inp["bg"].astype(np.float64), ex, w.k)
    np.testing.assert_allclose(res["out"], want, rtol=1e-12, atol=1e-12)


def check_sampled_tokens_match_full(seed=12):
    rng = np.random.default_rng(seed)
    x, Wg, ex = _rand_layer(rng, 80, 12, 16, 6)
    full = O.forward(x, Wg, None, None, 2, 1.0, 0.01, lambda e: ex[e])
    toks = np.array([79, 3, 40, 0, 41])
    part = O.forward(x, Wg, None, None, 2, 1.0, 0.01, lambda e: ex[e], tokens=toks)
    np.testing.assert_allclose(part["out"], full["out"][toks], rtol=0, atol=1e-15)


def check_empty_input():
    res = O.forward(np.zeros((0, 8)), np.ones((4, 8)), None, None, 2, 1.25, 0.01,
                    lambda e: (np.ones((6, 8)), None, np.ones((8, 6)), None))
    assert res["out"].shape == (0, 8)
    assert res["offsets"].tolist() == [0] * 5 and res["l_aux"] == 0.0
    assert res["capacity"] == 0


ALL_CHECKS = [
    check_router_worked_example, check_capacity_examples, check_permute_worked_example,
    check_laux_worked_examples, check_gelu_textbook, check_moelayer_worked_example,
    check_topk_bruteforce, check_router_vs_torch, check_selection_bias, check_zero_gate_all_ties,
    check_weights_invariants, check_permute_vs_stable_sort, check_dense_reduction,
    check_identical_experts, check_shared_only, check_linearity_in_w2, check_expert_relabelling,
    check_moelayer_restatement, check_tiny_workload_restatement, check_sampled_tokens_match_full,
    check_empty_input,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_pin(check):
    check()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail

def _mut_gelu_tanh(z):
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def _mut_renorm_no_division(P, idx):
    return np.take_along_axis(P, idx, axis=1)


def _mut_ties_high_index(s, k):
    s = np.asarray(s, np.float64)
    T, N = s.shape
    order = (N - 1 - np.argsort(-s[:, ::-1], axis=1, kind="stable"))
    return order[:, :k].copy(), np.full(T, np.inf), np.full(T, np.inf)


def _mut_capacity_ceil(T, N, cf):
    return None if cf <= 0 else int(math.ceil(T / N * cf))


def _mut_laux_no_n(P, counts, k, alpha):
    d = O.__dict__["_orig_load_balance"](P, counts, k, alpha)
    d["l_aux"] /= P.shape[1]
    return d


def _mut_bias_in_weights(x, Wg, bg, sel_bias, k):
    l = O.gate_logits(x, Wg, bg)
    s = l if sel_bias is None else l - np.asarray(sel_bias)[None, :]
    P = O.softmax(s)
    idx, margin, om = O.select_topk(s, k)
    return dict(logits=l, probs=O.softmax(l), idx=idx, w=O.renormalise(P, idx), margin=margin,
                order_margin=om, scores=s)


def _mut_ffn_missing_b2(xe, W1, b1, W2, b2):
    z = np.asarray(xe, np.float64) @ W1.T
    if b1 is not None:
        z = z + b1[None, :]
    return O.gelu(z) @ W2.T


def _mut_ffn_transposed_w2(xe, W1, b1, W2, b2):
    z = np.asarray(xe, np.float64) @ W1.T
    if b1 is not None:
        z = z + b1[None, :]
    g = O.gelu(z)
    y = g @ W2.T if W2.shape[0] != W2.shape[1] else g @ W2
    return y if b2 is None else y + b2[None, :]


def _mut_permute_keep_last(idx, N, C):
    """Keeps the last C assignments of each expert instead of the first C."""
    flat = np.asarray(idx).reshape(-1)
    rev = O.__dict__["_orig_permute"](flat[::-1].reshape(-1, 1), N, C)
    A = flat.shape[0]
    d = O.__dict__["_orig_permute"](idx, N, None)
    kept = rev["kept"]
    offsets = np.concatenate([[0], np.cumsum(kept)])
    perm = np.concatenate([np.sort(A - 1 - rev["perm"][rev["offsets"][e]:rev["offsets"][e + 1]])
                           for e in range(N)]).astype(np.int64)
    inv = np.full(A, -1)
    inv[perm] = np.arange(perm.shape[0])
    return dict(counts=d["counts"], kept=kept, offsets=offsets, perm=perm, inv=inv)


MUTANTS = {
    "gelu_tanh_approx": ("gelu", _mut_gelu_tanh),
    "renorm_dropped": ("renormalise", _mut_renorm_no_division),
    "ties_to_high_index": ("select_topk", _mut_ties_high_index),
    "capacity_ceil": ("capacity", _mut_capacity_ceil),
    "laux_missing_N": ("load_balance", _mut_laux_no_n),
    "sel_bias_in_weights": ("route", _mut_bias_in_weights),
    "ffn_missing_b2": ("expert_ffn", _mut_ffn_missing_b2),
    "ffn_w2_transposed": ("expert_ffn", _mut_ffn_transposed_w2),
    "drop_first_not_last": ("permute", _mut_permute_keep_last),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setitem(O.__dict__, "_orig_" + name, getattr(O, name))
    monkeypatch.setattr(O, name, fn)
    failed = []
    for check in ALL_CHECKS:
        try:
            check()
        except Exception:  # noqa: BLE001 - any failure counts as detection
            failed.append(check.__name__)
    assert failed, f"no pin detects the planted mistake {mutant}"
