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

Widened rows (the pages name them; each reading is a choice):

* drop order: "token" (default, above) or "slot": every token's first
  choice claims slots before any second choice, and so on.
* min_capacity ([SKILLS] §5.1's DeepSpeed block): raises a smaller capacity
  to the floor; it does not apply without a capacity factor.
* SiLU / SwiGLU ([SKILLS] §6.1 prints a two-Linear SiLU expert while its text
  says SwiGLU): "silu" is the printed block; "swiglu" keeps W1 as [2F, H]
  with the gate rows first and the up rows second, SiLU(gate) * up.
* expert choice ([SKILLS] §4.2, §7.3): selection on the router logits as
  printed (router(x) transposed, top-k along tokens), ties to the lower
  token; the combining weight is the token's gate probability P[t, e]
  (softmax over experts), not renormalised; C = the capacity formula capped
  at T; the selection bias is not used.
* router z-loss ([SKILLS] §4.3): the raw mean of logsumexp(l_t)^2.
* auxiliary-loss-free bias step ([ARCH] §2.4): b_i += gamma * sign(count_i -
  mean count); the pages give no rate, so gamma is an input.
* FP8 weights (the inference guide's "FP8 量化"): the pages name FP8 and its
  gains, not a format; read as E4M3 codes with one fp32 scale per output
  row of each weight matrix, dequantised exactly before the Linears;
  activations stay as they are.

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

def capacity(T: int, N: int, capacity_factor: float, min_capacity: int = 0) -> Optional[int]:
    """Capacity = floor(T / N * capacity_factor); None (no limit) when cf <= 0.

    ``min_capacity`` is the DeepSpeed ``moe`` block's floor ([SKILLS] §5.1):
    the capacity is raised to it when the formula gives less."""
    if capacity_factor <= 0:
        return None
    c = int(math.floor(float(T) / float(N) * float(capacity_factor)))
    return max(c, int(min_capacity))


def claim_order(T: int, k: int, order: str = "token") -> np.ndarray:
    """The order in which the T*k assignments a = t*k + j claim expert slots.

    "token": increasing a (token by token, a token's slots in rank order);
    "slot": every token's first choice, then every token's second choice,
    and so on (a = t*k + j for j-major, then t).
    """
    if order == "token":
        return np.arange(T * k, dtype=np.int64)
    if order == "slot":
        return np.array([t * k + j for j in range(k) for t in range(T)], dtype=np.int64)
    raise ValueError(order)


def permute(idx: np.ndarray, N: int, C: Optional[int], order: str = "token") -> dict:
    """Stable, capacity-limited dispatch of the T*k assignments to experts.

    Walks the assignments in claim_order(order) with one counter per expert.
    An assignment whose rank within its expert is below C gets row
    offsets[e] + rank in the expert-contiguous layout; the rest are dropped.

    Returns counts [N] (before drops), kept [N], offsets [N+1],
    perm [R] (row -> a) and inv [T*k] (a -> row, or -1 if dropped).
    """
    idx = np.asarray(idx)
    flat = idx.reshape(-1)
    A = flat.shape[0]
    T, k = (idx.shape[0], idx.shape[1]) if idx.ndim == 2 else (A, 1)
    counts = np.zeros(N, np.int64)
    rank = np.empty(A, np.int64)
    for a in claim_order(T, k, order):
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
# router z-loss: [SKILLS] §4.3

def z_loss(l: np.ndarray) -> float:
    """mean over tokens of logsumexp(l_t)^2 (the raw statistic; the pages
    weight it by 0.001 in the training loss).  0 for T = 0."""
    l = np.asarray(l, np.float64)
    if l.shape[0] == 0:
        return 0.0
    m = l.max(axis=1)
    lse = m + np.log(np.exp(l - m[:, None]).sum(axis=1))
    return float(np.mean(lse * lse))


# ---------------------------------------------------------------------------
# auxiliary-loss-free balancing step: [ARCH] §2.4

def update_sel_bias(b: np.ndarray, counts: np.ndarray, gamma: float) -> np.ndarray:
    """b_i + gamma * sign(count_i - mean count): the bias of an expert that
    took more than its share of assignments rises (it is subtracted from the
    logits for selection, so it is chosen less), that of one that took less
    falls, and an expert at exactly the mean keeps its bias.  The pages give
    no rate; gamma is the caller's."""
    c = np.asarray(counts, np.float64)
    mean = c.sum() / c.shape[0]
    return np.asarray(b, np.float64) + gamma * np.sign(c - mean)


# ---------------------------------------------------------------------------
# expert-choice routing: [SKILLS] §4.2 and §7.3

def expert_choice(l: np.ndarray, C: int) -> dict:
    """Each expert takes the C tokens with the largest router logits in its
    column (router(x) transposed, top-k along tokens); equal logits take the
    lower token index first.  C is capped at T.

    Rows: expert e owns rows [e*C, (e+1)*C), its tokens in increasing token
    order.  Assignment ids are a = t*N + e.  Returns offsets [N+1],
    perm [N*C] (row -> a), inv [T*N] (a -> row or -1), counts [N] and the
    column margins: for each expert, the logit gap between its C-th and
    (C+1)-th token (+inf when C == T), which flags selections that a tiny
    change of the logits can flip.
    """
    l = np.asarray(l, np.float64)
    T, N = l.shape
    C = min(int(C), T)
    offsets = np.arange(N + 1, dtype=np.int64) * C
    perm = np.empty(N * C, np.int64)
    inv = np.full(T * N, -1, np.int64)
    margin = np.full(N, np.inf)
    for e in range(N):
        order = np.argsort(-l[:, e], kind="stable")   # ties: lower token first
        chosen = np.sort(order[:C])
        if C < T:
            margin[e] = l[order[C - 1], e] - l[order[C], e]
        for r, t in enumerate(chosen):
            perm[e * C + r] = t * N + e
            inv[t * N + e] = e * C + r
    return dict(offsets=offsets, perm=perm, inv=inv, counts=np.full(N, C, np.int64),
                kept=np.full(N, C, np.int64), ec_margin=margin)


# ---------------------------------------------------------------------------
# FP8 expert weights ([SKILLS] §9.2, "FP8 量化" of the inference guide):
# E4M3 codes with one fp32 scale per output row

def e4m3_decode(bits: np.ndarray) -> np.ndarray:
    """Value of FP8 E4M3 codes: sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; exponent field 0 holds the subnormals m * 2^-9; there is no
    infinity and the all-ones pattern is NaN."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[r, :] = scale[r] * decode(codes[r, :]), exactly in float64."""
    return e4m3_decode(codes) * np.asarray(scales, np.float64).reshape(-1, 1)


# ---------------------------------------------------------------------------
# experts: [SKILLS] §3.1 (Linear(H,F) -> GELU -> Linear(F,H))

def gelu(z: np.ndarray) -> np.ndarray:
    """Exact GELU: z * Phi(z) = 0.5 * z * (1 + erf(z / sqrt(2)))."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU (the Mixtral block's nn.SiLU, [SKILLS] §6.1): z * sigmoid(z),
    written z / (1 + exp(-z)) for z >= 0 and z * exp(z) / (1 + exp(z)) below,
    so that neither branch overflows."""
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


ACTIVATIONS = ("gelu", "silu", "swiglu")


def expert_ffn(xe, W1, b1, W2, b2, activation: str = "gelu") -> np.ndarray:
    """y = W2 . act(W1 . x + b1) + b2 for the rows of xe ([rows, H]).

    "gelu": [SKILLS] §3.1's Linear(H, F) -> GELU -> Linear(F, H).
    "silu": the two-Linear SiLU expert printed in [SKILLS] §6.1.
    "swiglu": the gated form that §6.1's text names for Mixtral: W1 holds the
    gate rows [0, F) and the up rows [F, 2F) (b1 likewise), and
    act(z) = SiLU(z_gate) * z_up.
    """
    z = np.asarray(xe, np.float64) @ W1.T
    if b1 is not None:
        z = z + b1[None, :]
    if activation == "gelu":
        h = gelu(z)
    elif activation == "silu":
        h = silu(z)
    elif activation == "swiglu":
        F = z.shape[1] // 2
        h = silu(z[:, :F]) * z[:, F:]
    else:
        raise ValueError(activation)
    y = h @ W2.T
    if b2 is not None:
        y = y + b2[None, :]
    return y


# ---------------------------------------------------------------------------
# the whole layer: [SKILLS] §3.1 / §6.1 / §7.1, [ARCH] §3

def forward(x, Wg, bg, sel_bias, k: int, capacity_factor: float, alpha: float,
            expert: Callable[[int], tuple], shared: Optional[tuple] = None,
            tokens: Optional[np.ndarray] = None, routing: str = "token",
            activation: str = "gelu", min_capacity: int = 0,
            drop_order: str = "token") -> dict:
    """Forward pass of one sparse MoE FFN layer.

    ``expert(e)`` returns float64 (W1 [F,H] ([2F,H] for swiglu), b1|None,
    W2 [H,F], b2 [H]|None) of routed expert e; ``shared`` is the same tuple
    for the always-on shared expert (same activation), or None.  Routing,
    capacity and the statistics always cover all T tokens; with ``tokens``
    given, the expert outputs are evaluated only for those rows (``out`` then
    has one row per listed token, in that order).

    routing "token" (token choice, [SKILLS] §3.1):
        out[t] = sum over kept slots j of w_tj * FFN_{idx_tj}(x_t)  (+ FFN_s(x_t))
    routing "expert" (expert choice, [SKILLS] §4.2): expert e takes the
    C = capacity(T, N, cf, min_capacity) tokens with the largest logits l[:, e];
        out[t] = sum over experts e that took t of P[t, e] * FFN_e(x_t)  (+ FFN_s(x_t))
    with P the gate softmax (the same gate probability the token-choice
    weights come from; not renormalised, since a token may be taken by any
    number of experts).  The selection bias does not apply.
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    N = np.asarray(Wg).shape[0]
    if routing == "token":
        r = route(x, Wg, bg, sel_bias, k)
        C = capacity(T, N, capacity_factor, min_capacity)
        d = permute(r["idx"], N, C, drop_order)
        lb = load_balance(r["probs"], d["counts"], k, alpha)
        k_slots = k
        weight_of = lambda a: r["w"][a // k, a % k]   # noqa: E731
    elif routing == "expert":
        l = gate_logits(x, Wg, bg)
        P = softmax(l)
        r = dict(logits=l, probs=P)
        C = capacity(T, N, capacity_factor, min_capacity)
        if C is None:
            raise ValueError("expert choice needs a capacity factor > 0")
        d = expert_choice(l, C)
        # every expert takes the same number of tokens: f_i = 1/N
        tot = max(int(d["counts"].sum()), 1)
        f = d["counts"] / tot
        p = P.mean(axis=0) if T > 0 else np.zeros(N)
        lb = dict(f=f, p=p, l_aux=float(alpha * N * np.sum(f * p)))
        k_slots = N
        weight_of = lambda a: P[a // N, a % N]   # noqa: E731
    else:
        raise ValueError(routing)
    z = z_loss(r["logits"])

    rows_out = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    where = np.full(T, -1, np.int64)
    where[rows_out] = np.arange(rows_out.shape[0])
    H = x.shape[1]
    out = np.zeros((rows_out.shape[0], H), np.float64)
    offsets, perm = d["offsets"], d["perm"]
    for e in range(N):
        a = perm[offsets[e]:offsets[e + 1]]
        t = a // k_slots
        keep = where[t] >= 0
        a, t = a[keep], t[keep]
        if a.shape[0] == 0:
            continue
        W1, b1, W2, b2 = expert(e)
        y = expert_ffn(x[t], W1, b1, W2, b2, activation)
        wt = weight_of(a)
        # one writer per assignment: each appears once in perm
        np.add.at(out, where[t], wt[:, None] * y)
    if shared is not None:
        W1s, b1s, W2s, b2s = shared
        out += expert_ffn(x[rows_out], W1s, b1s, W2s, b2s, activation)
    res = dict(out=out, capacity=C, z_loss=z, **r, **d, **lb)
    return res
