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


# ---------------------------------------------------------------------------
# widened rows: drop order, min_capacity, SiLU / SwiGLU, expert choice,
# router z-loss, aux-loss-free bias step

def check_slot_major_worked_example():
    g = _golden("permute_slot_major_example.json")
    idx = np.asarray(g["idx"])
    for key in ("capped", "unlimited"):
        c = g[key]
        C = O.capacity(g["T"], g["N"], c["cf"])
        d = O.permute(idx, g["N"], C, "slot")
        assert d["counts"].tolist() == g["counts"]
        for f in ("kept", "offsets", "perm", "inv"):
            assert d[f].tolist() == c[f], (key, f, d[f].tolist())


def check_min_capacity_examples():
    for c in _golden("min_capacity_examples.json")["cases"]:
        assert O.capacity(c["T"], c["N"], c["cf"], c["min"]) == c["C"], c


def check_slot_major_vs_stable_sort(seed=13):
    """Slot-major dispatch = a stable sort of the assignments by expert after
    reordering them j-major (numpy's stable argsort as the reference)."""
    rng = np.random.default_rng(seed)
    for T, k, N, C in [(37, 3, 5, 9), (50, 2, 4, None), (20, 4, 6, 3)]:
        idx = np.stack([rng.permutation(N)[:k] for _ in range(T)])
        d = O.permute(idx, N, C, "slot")
        order = np.array([t * k + j for j in range(k) for t in range(T)])
        e_of = idx.reshape(-1)[order]
        srt = order[np.argsort(e_of, kind="stable")]
        rows = []
        for e in range(N):
            a_e = srt[idx.reshape(-1)[srt] == e]
            rows.extend(a_e[:C] if C is not None else a_e)
        assert d["perm"].tolist() == [int(a) for a in rows]


def check_silu_textbook():
    z = np.array([-800.0, -50.0, -3.0, -1.0, -1e-3, 0.0, 1e-3, 0.5, 2.0, 40.0, 800.0])
    s_ = O.silu(z)
    assert np.all(np.isfinite(s_)) and s_[5] == 0.0
    # z*sigmoid(z) - (-z)*sigmoid(-z) = z (sigmoid(z) + sigmoid(-z) = 1)
    np.testing.assert_allclose(s_ - O.silu(-z), z, rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(s_[-1], 800.0, rtol=1e-15)
    assert abs(s_[0]) < 1e-300
    rng = np.random.default_rng(14)
    r = rng.normal(0, 4, size=500)
    np.testing.assert_allclose(O.silu(r), TF.silu(torch.from_numpy(r)).numpy(), rtol=1e-14,
                               atol=1e-300)


def check_swiglu_structure(seed=15):
    rng = np.random.default_rng(seed)
    H, F = 12, 10
    x = rng.normal(size=(7, H))
    Wg, Wu, Wu2 = (rng.normal(size=(F, H)) for _ in range(3))
    W2, b2 = rng.normal(size=(H, F)), rng.normal(size=H)
    ffn = lambda gate, up, b1=None: O.expert_ffn(x, np.vstack([gate, up]), b1, W2, b2, "swiglu")  # noqa: E731
    # a zero gate switches the expert off: SiLU(0) = 0
    np.testing.assert_allclose(ffn(np.zeros((F, H)), Wu), np.tile(b2, (7, 1)), rtol=0, atol=0)
    # linear in the up projection (and only there)
    lin = ffn(Wg, Wu + Wu2) - b2
    np.testing.assert_allclose(lin, (ffn(Wg, Wu) - b2) + (ffn(Wg, Wu2) - b2), rtol=1e-12,
                               atol=1e-12)
    assert not np.allclose(ffn(Wg + Wu2, Wu) - b2, (ffn(Wg, Wu) - b2) + (ffn(Wu2, Wu) - b2))
    # one hidden unit by hand: gate row g, up row u -> silu(g.x) * (u.x) * W2[:, 0]
    g1, u1 = np.zeros((F, H)), np.zeros((F, H))
    g1[0, 0], u1[0, 1] = 1.0, 1.0
    want = (O.silu(x[:, 0]) * x[:, 1])[:, None] * W2[:, 0][None, :] + b2
    np.testing.assert_allclose(ffn(g1, u1), want, rtol=1e-13, atol=1e-13)
    # the plain SiLU expert is the GELU expert with the activation swapped
    z = x @ Wg.T
    np.testing.assert_allclose(O.expert_ffn(x, Wg, None, W2, None, "silu"),
                               TF.silu(torch.from_numpy(z)).numpy() @ W2.T, rtol=1e-12,
                               atol=1e-12)


def _ec_bruteforce(l, C):
    """Per expert, the lexicographically first C-subset of tokens with the
    largest logit sum (itertools.combinations enumerates in lexicographic
    order, so the first maximum wins): top-C with ties to lower tokens."""
    T, N = l.shape
    out = []
    for e in range(N):
        best, best_set = -np.inf, None
        for comb in itertools.combinations(range(T), C):
            v = sum(l[t, e] for t in comb)
            if v > best:
                best, best_set = v, comb
        out.append(list(best_set))
    return out


def check_expert_choice_bruteforce(seed=16):
    rng = np.random.default_rng(seed)
    for T, N, C in [(6, 3, 2), (7, 2, 3), (5, 4, 5), (6, 2, 1)]:
        for ties in (False, True):
            l = rng.integers(-2, 3, size=(T, N)).astype(np.float64) if ties else \
                rng.normal(size=(T, N))
            d = O.expert_choice(l, C)
            want = _ec_bruteforce(l, C)
            for e in range(N):
                a = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
                assert (a // N).tolist() == want[e], (T, N, C, ties, e)
                assert np.all(a % N == e)


def check_expert_choice_invariants(seed=17):
    rng = np.random.default_rng(seed)
    T, N = 40, 5
    l = rng.normal(size=(T, N))
    for C in (1, 7, 40, 60):
        d = O.expert_choice(l, C)
        Ce = min(C, T)
        assert d["offsets"].tolist() == [e * Ce for e in range(N + 1)]
        assert np.all(d["inv"][d["perm"]] == np.arange(N * Ce))
        assert int((d["inv"] >= 0).sum()) == N * Ce
        for e in range(N):
            toks = d["perm"][e * Ce:(e + 1) * Ce] // N
            assert np.all(np.diff(toks) > 0)
            rest = np.setdiff1d(np.arange(T), toks)
            if rest.size:
                assert l[toks, e].min() >= l[rest, e].max()


def check_expert_choice_full_capacity(seed=18):
    """C = T: every expert takes every token, so with identical experts the
    layer is the dense FFN (the gate probabilities of a token sum to one)."""
    rng = np.random.default_rng(seed)
    T, H, F, N = 9, 6, 8, 3
    x, Wg, ex = _rand_layer(rng, T, H, F, N)
    bg = rng.normal(size=N)
    same = ex[0]
    res = O.forward(x, Wg, bg, None, 1, float(N), 0.01, lambda e: same, routing="expert")
    assert res["capacity"] == T
    np.testing.assert_allclose(res["out"], O.expert_ffn(x, *same), rtol=1e-12, atol=1e-12)
    # and a token nobody takes gets zero: C = 1 on distinct experts
    res1 = O.forward(x, Wg, bg, None, 1, N / T, 0.01, lambda e: ex[e], routing="expert")
    taken = set((res1["perm"] // N).tolist())
    for t in range(T):
        if t not in taken:
            assert np.all(res1["out"][t] == 0.0)


def check_z_loss(seed=19):
    from scipy.special import logsumexp
    for c, N in [(0.0, 4), (2.5, 8), (-3.0, 256)]:
        np.testing.assert_allclose(O.z_loss(np.full((5, N), c)), (c + math.log(N)) ** 2,
                                   rtol=1e-14)
    l = np.random.default_rng(seed).normal(0, 3, size=(50, 16))
    np.testing.assert_allclose(O.z_loss(l), np.mean(logsumexp(l, axis=1) ** 2), rtol=1e-13)
    assert O.z_loss(np.zeros((0, 4))) == 0.0


def check_update_sel_bias():
    # mean count 4: the over-used expert 0 rises, the under-used expert 1 falls
    b = O.update_sel_bias(np.array([0.1, -0.2, 0.0, 0.3]), np.array([5, 3, 4, 4]), 0.01)
    np.testing.assert_allclose(b, [0.11, -0.21, 0.0, 0.3], rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.update_sel_bias(np.zeros(3), np.array([2, 2, 2]), 1.0),
                               [0.0, 0.0, 0.0])


def check_e4m3_decode():
    """E4M3 decode against hand values of the format and against torch's
    float8_e4m3fn (a library routine), all 256 codes."""
    hand = {0x00: 0.0, 0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6,
            0x3A: 1.25, 0xC0: -2.0, 0x07: 7 * 2.0 ** -9, 0x77: 240.0}
    for b, v in hand.items():
        assert O.e4m3_decode(np.array([b]))[0] == v, (hex(b), v)
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # per-row scaling
    q = np.array([[0x38, 0xC0], [0x7E, 0x00]], dtype=np.uint8)
    np.testing.assert_array_equal(O.dequantize_rows(q, np.array([0.5, 2.0])),
                                  [[0.5, -1.0], [896.0, 0.0]])


ALL_CHECKS = [
    check_router_worked_example, check_capacity_examples, check_permute_worked_example,
    check_laux_worked_examples, check_gelu_textbook, check_moelayer_worked_example,
    check_topk_bruteforce, check_router_vs_torch, check_selection_bias, check_zero_gate_all_ties,
    check_weights_invariants, check_permute_vs_stable_sort, check_dense_reduction,
    check_identical_experts, check_shared_only, check_linearity_in_w2, check_expert_relabelling,
    check_moelayer_restatement, check_tiny_workload_restatement, check_sampled_tokens_match_full,
    check_empty_input, check_slot_major_worked_example, check_min_capacity_examples,
    check_slot_major_vs_stable_sort, check_silu_textbook, check_swiglu_structure,
    check_expert_choice_bruteforce, check_expert_choice_invariants,
    check_expert_choice_full_capacity, check_z_loss, check_update_sel_bias, check_e4m3_decode,
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


def _mut_capacity_ceil(T, N, cf, min_capacity=0):
    return None if cf <= 0 else max(int(math.ceil(T / N * cf)), min_capacity)


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


def _mut_ffn_missing_b2(xe, W1, b1, W2, b2, activation="gelu"):
    y = O.__dict__["_orig_expert_ffn"](xe, W1, b1, W2, None, activation)
    return y


def _mut_ffn_transposed_w2(xe, W1, b1, W2, b2, activation="gelu"):
    W2m = W2 if W2.shape[0] != W2.shape[1] else W2.T
    return O.__dict__["_orig_expert_ffn"](xe, W1, b1, W2m, b2, activation)


def _mut_permute_keep_last(idx, N, C, order="token"):
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


def _mut_min_capacity_ignored(T, N, cf, min_capacity=0):
    return O.__dict__["_orig_capacity"](T, N, cf)


def _mut_slot_order_ignored(T, k, order="token"):
    return np.arange(T * k, dtype=np.int64)


def _mut_silu_is_sigmoid(z):
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(-np.clip(z, -700, 700)))


def _mut_swiglu_halves_swapped(xe, W1, b1, W2, b2, activation="gelu"):
    if activation == "swiglu":
        F = W1.shape[0] // 2
        W1 = np.vstack([W1[F:], W1[:F]])
        if b1 is not None:
            b1 = np.concatenate([b1[F:], b1[:F]])
    return O.__dict__["_orig_expert_ffn"](xe, W1, b1, W2, b2, activation)


def _mut_ec_ties_high_token(l, C):
    l = np.asarray(l, np.float64)
    T = l.shape[0]
    d = O.__dict__["_orig_expert_choice"](l[::-1], C)
    N = l.shape[1]
    perm = d["perm"].copy()
    for e in range(N):
        seg = perm[d["offsets"][e]:d["offsets"][e + 1]]
        toks = np.sort(T - 1 - seg // N)
        perm[d["offsets"][e]:d["offsets"][e + 1]] = toks * N + e
    inv = np.full(T * N, -1)
    inv[perm] = np.arange(perm.shape[0])
    return dict(d, perm=perm, inv=inv)


def _mut_zloss_no_square(l):
    l = np.asarray(l, np.float64)
    if l.shape[0] == 0:
        return 0.0
    m = l.max(axis=1)
    return float(np.mean(m + np.log(np.exp(l - m[:, None]).sum(axis=1))))


def _mut_bias_update_sign(b, counts, gamma):
    return O.__dict__["_orig_update_sel_bias"](b, counts, -gamma)


def _mut_e4m3_bias8(bits):
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e, m = (b >> 3) & 0xF, b & 0x7
    return sign * np.where(e == 0, m * 2.0 ** -10, (1.0 + m / 8.0) * np.exp2(e - 8.0))


MUTANTS = {
    "e4m3_exponent_bias_8": ("e4m3_decode", _mut_e4m3_bias8),
    "min_capacity_ignored": ("capacity", _mut_min_capacity_ignored),
    "slot_major_as_token_major": ("claim_order", _mut_slot_order_ignored),
    "silu_as_sigmoid": ("silu", _mut_silu_is_sigmoid),
    "swiglu_gate_up_swapped": ("expert_ffn", _mut_swiglu_halves_swapped),
    "expert_choice_ties_high_token": ("expert_choice", _mut_ec_ties_high_token),
    "z_loss_not_squared": ("z_loss", _mut_zloss_no_square),
    "bias_update_sign_flipped": ("update_sel_bias", _mut_bias_update_sign),
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
