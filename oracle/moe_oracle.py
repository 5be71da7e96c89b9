"""Plain, slow CPU oracle of the sparse Mixture-of-Experts FFN forward pass.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The CUDA library shares no code
with it and never calls it.

Everything is float64 numpy, written as the pages define each step, one
step per function; a matrix product (``@``) and ``erf`` are the only library
primitives used.  Sources (page title, section):

* "AI-Research-SKILLs MoE 训练实战：稀疏专家模型的架构、路由、负载均衡与推理优化全指南"
  (cited below as [SKILLS]): §3.1 the MoELayer (gate Linear with bias ->
  softmax -> top-k -> renormalise -> per-expert Linear->GELU->Linear ->
  weighted sum); §4.3 the load-balancing loss; §6.1 the Mixtral block
  (per-expert gather and index_add combine); §7.1 DeepSeekMoE (shared
  expert added to the routed sum); §8.2 the capacity formula.
* "混合专家模型 MoE 架构深度解析：从路由机制到生产级推理部署" (cited below
  as [ARCH]): §1.2 gate formula; §1.3 the four-step top-K algorithm; §2.2
  L_aux = alpha*N*sum(f_i*p_i); §2.3 Capacity = floor(T/N * capacity_factor)
  with overflow tokens passing through with no expert output; §2.4 the
  per-expert bias b_i subtracted from the logits for selection; §3 the
  shared expert, Output = Shared(x) + sum_j w_j Routed_j(x).

Readings where the pages are silent or disagree (each is a choice, not a
quote):

* selection bias: subtracted from the logits and used for selection only;
  the weights come from the unbiased softmax, renormalised over the k
  chosen experts ([ARCH] §2.4 over the [SKILLS] §4.3 variant that adds it).
* selection is made on the scores s = l - b directly (softmax is monotone, so
  this is the same ranking as top-k of probabilities, without rounding ties).
* ties: equal scores rank the lower expert index first; the k slots of a
  token are in descending score order.  Tokens whose k-th and (k+1)-th
  selection probabilities are within 1e-5 (the set can flip) or whose
  adjacent slots inside the top k are within 1e-5 (the slot order can flip)
  are flagged by the margins select_topk returns.
* capacity: floor(T / N * cf) evaluated in double in that order;
  cf <= 0 means no limit.  Assignments a = t*k + j claim slots in increasing
  a; an assignment whose rank within its expert is >= C is dropped and
  contributes zero; the surviving weights are not renormalised.
* f_i counts assignments before capacity drops over T*k ([SKILLS] §4.3
  bincount / numel); p_i is the mean over tokens of the full unbiased
  softmax (gate bias included, selection bias not).
* GELU is the exact erf form (nn.GELU default).
* T = 0: no outputs, f = p = 0 and L_aux = 0.

Parity pins for every function live in the tests (closed forms, brute force,
textbook routines, hand-worked fixtures); none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Callable, Optional

import numpy as np
from scipy.special import erf as _erf


# ---------------------------------------------------------------------------
# router: [ARCH] §1.2, §1.3, §2.4; [SKILLS] §3.1

def gate_logits(x: np.ndarray, Wg: np.ndarray, bg: Optional[np.ndarray] = None) -> np.ndarray:
    """l = x . W_g^T (+ b_g): the gate Linear of [SKILLS] §3.1 / [ARCH] §1.2.

    ``Wg`` is stored [N, H] (nn.Linear layout), the transpose of the
    [d_model, N_experts] matrix drawn in [ARCH] §1.2; the product is the same.
    """
    l = np.asarray(x, np.float64) @ np.asarray(Wg, np.float64).T
    if bg is not None:
        l = l + np.asarray(bg, np.float64)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    """Row softmax over the N experts (max-subtracted for range)."""
    l = np.asarray(l, np.float64)
    if l.shape[0] == 0:
        return l.copy()
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def select_topk(s: np.ndarray, k: int):
    """[ARCH] §1.3 step 2: the k experts with the largest scores.

    Returns (idx int64 [T,k] in descending score order, ties to the lower
    index; margin float64 [T] = q_k - q_{k+1} where q = softmax(s) sorted
    descending, +inf when k == N; order_margin float64 [T] = the smallest
    gap q_j - q_{j+1} for j < k, +inf when k == 1).  The margin flags tokens
    whose chosen set a tiny change of the scores can flip; the order margin
    flags tokens whose slot order it can flip.
    """
    s = np.asarray(s, np.float64)
    T, N = s.shape
    order = np.argsort(-s, axis=1, kind="stable")
    idx = order[:, :k].copy()
    if T == 0:
        return idx, np.full(T, np.inf), np.full(T, np.inf)
    q = np.take_along_axis(softmax(s), order, axis=1)
    margin = q[:, k - 1] - q[:, k] if k < N else np.full(T, np.inf)
    order_margin = (-np.diff(q[:, :k], axis=1)).min(axis=1) if k > 1 else np.full(T, np.inf)
    return idx, margin, order_margin


def renormalise(P: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """[ARCH] §1.3 step 3 / [SKILLS] §3.1: w_tj = P[t, idx_tj] / sum_j' P[t, idx_tj']."""
    sel = np.take_along_axis(P, idx, axis=1)
    if sel.shape[0] == 0:
        return sel
    return sel / sel.sum(axis=1, keepdims=True)


def route(x, Wg, bg, sel_bias, k: int) -> dict:
    """Gate -> softmax -> top-k on (l - b_sel) -> renormalised weights."""
    l = gate_logits(x, Wg, bg)
    P = softmax(l)
    s = l if sel_bias is None else l - np.asarray(sel_bias, np.float64)[None, :]
    idx, margin, order_margin = select_topk(s, k)
    w = renormalise(P, idx)
    return dict(logits=l, probs=P, idx=idx, w=w, margin=margin, order_margin=order_margin,
                scores=s)


# ---------------------------------------------------------------------------
# dispatch: [ARCH] §2.3, [SKILLS] §8.2 (capacity) and §4.4 (drop_tokens)

def capacity(T: int, N: int, capacity_factor: float) -> Optional[int]:
    """Capacity = floor(T / N * capacity_factor); None (no limit) when cf <= 0."""
    if capacity_factor <= 0:
        return None
    return int(math.floor(float(T) / float(N) * float(capacity_factor)))


def permute(idx: np.ndarray, N: int, C: Optional[int]) -> dict:
    """Stable, capacity-limited dispatch of the T*k assignments to experts.

    Walks the assignments a = t*k + j in increasing a with one counter per
    expert.  An assignment whose rank within its expert is below C gets row
    offsets[e] + rank in the expert-contiguous layout; the rest are dropped.

    Returns counts [N] (before drops), kept [N], offsets [N+1],
    perm [R] (row -> a) and inv [T*k] (a -> row, or -1 if dropped).
    """
    flat = np.asarray(idx).reshape(-1)
    A = flat.shape[0]
    counts = np.zeros(N, np.int64)
    rank = np.empty(A, np.int64)
    for a in range(A):
        e = int(flat[a])
        rank[a] = counts[e]
        counts[e] += 1
    kept = counts.copy() if C is None else np.minimum(counts, C)
    offsets = np.zeros(N + 1, np.int64)
    offsets[1:] = np.cumsum(kept)
    perm = np.empty(int(offsets[-1]), np.int64)
    inv = np.full(A, -1, np.int64)
    for a in range(A):
        e = int(flat[a])
        if C is None or rank[a] < C:
            row = offsets[e] + rank[a]
            perm[row] = a
            inv[a] = row
    return dict(counts=counts, kept=kept, offsets=offsets, perm=perm, inv=inv)


# ---------------------------------------------------------------------------
# load-balance statistic: [ARCH] §2.2, [SKILLS] §4.3

def load_balance(P: np.ndarray, counts: np.ndarray, k: int, alpha: float) -> dict:
    """f_i = count_i / (T*k), p_i = mean_t P[t,i], L_aux = alpha * N * sum_i f_i p_i."""
    T, N = P.shape
    if T == 0:
        z = np.zeros(N)
        return dict(f=z, p=z.copy(), l_aux=0.0)
    f = np.asarray(counts, np.float64) / float(T * k)
    p = P.mean(axis=0)
    return dict(f=f, p=p, l_aux=float(alpha * N * np.sum(f * p)))


# ---------------------------------------------------------------------------
# experts: [SKILLS] §3.1 (Linear(H,F) -> GELU -> Linear(F,H))

def gelu(z: np.ndarray) -> np.ndarray:
    """Exact GELU: z * Phi(z) = 0.5 * z * (1 + erf(z / sqrt(2)))."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def expert_ffn(xe, W1, b1, W2, b2) -> np.ndarray:
    """y = W2 . GELU(W1 . x + b1) + b2 for the rows of xe ([rows, H])."""
    z = np.asarray(xe, np.float64) @ W1.T
    if b1 is not None:
        z = z + b1[None, :]
    y = gelu(z) @ W2.T
    if b2 is not None:
        y = y + b2[None, :]
    return y


# ---------------------------------------------------------------------------
# the whole layer: [SKILLS] §3.1 / §6.1 / §7.1, [ARCH] §3

def forward(x, Wg, bg, sel_bias, k: int, capacity_factor: float, alpha: float,
            expert: Callable[[int], tuple], shared: Optional[tuple] = None,
            tokens: Optional[np.ndarray] = None) -> dict:
    """Forward pass of one sparse MoE FFN layer.

    ``expert(e)`` returns float64 (W1 [F,H], b1 [F]|None, W2 [H,F], b2 [H]|None)
    of routed expert e; ``shared`` is the same tuple for the always-on shared
    expert, or None.  Routing, capacity and the statistics always cover all T
    tokens; with ``tokens`` given, the expert outputs are evaluated only for
    those rows (``out`` then has one row per listed token, in that order).

    out[t] = sum over kept slots j of w_tj * FFN_{idx_tj}(x_t)  (+ FFN_s(x_t))
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    N = np.asarray(Wg).shape[0]
    r = route(x, Wg, bg, sel_bias, k)
    C = capacity(T, N, capacity_factor)
    d = permute(r["idx"], N, C)
    lb = load_balance(r["probs"], d["counts"], k, alpha)

    rows_out = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    where = np.full(T, -1, np.int64)
    where[rows_out] = np.arange(rows_out.shape[0])
    H = x.shape[1]
    out = np.zeros((rows_out.shape[0], H), np.float64)
    offsets, perm = d["offsets"], d["perm"]
    for e in range(N):
        a = perm[offsets[e]:offsets[e + 1]]
        t = a // k
        keep = where[t] >= 0
        a, t = a[keep], t[keep]
        if a.shape[0] == 0:
            continue
        W1, b1, W2, b2 = expert(e)
        y = expert_ffn(x[t], W1, b1, W2, b2)
        wt = r["w"][t, a % k]
        # one writer per (t, j): each assignment appears once in perm
        np.add.at(out, where[t], wt[:, None] * y)
    if shared is not None:
        W1s, b1s, W2s, b2s = shared
        out += expert_ffn(x[rows_out], W1s, b1s, W2s, b2s)
    res = dict(out=out, capacity=C, **r, **d, **lb)
    return res
