"""Seeded synthetic workloads for the sparse MoE FFN forward pass.

This module only makes input data: shapes of the named workloads and seeded
random tensors.  It holds none of the layer's arithmetic, so both the CPU
oracle (through the tests) and the CUDA path (through the tests and the
benchmark) can take their inputs from it.

Seed tree
---------
Every tensor block is drawn from its own PCG64 stream,
``SeedSequence(entropy=seed, spawn_key=(tensor_id, block))``, where
``block`` is the expert index for per-expert tensors, the row-chunk index
(``X_CHUNK_ROWS`` rows per chunk) for the activations, and 0 otherwise.
A block's values therefore do not depend on which other blocks are drawn,
on the order of drawing or on the number of threads; the oracle can
regenerate the handful of experts a sampled token needs without drawing
the rest.

Values are drawn in float32 and, for the bf16 tensors, rounded to bf16 with
round-to-nearest-even; the bf16 tensors are returned as their uint16 bit
patterns so that the oracle and the GPU read identical bytes.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Callable, Dict, Optional

import numpy as np

X_CHUNK_ROWS = 4096
_TENSOR_ID = {
    "x": 0, "Wg": 1, "bg": 2, "sel_bias": 3,
    "W1": 4, "b1": 5, "W2": 6, "b2": 7,
    "W1s": 8, "b1s": 9, "W2s": 10, "b2s": 11,
}


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic MoE layer workload."""
    name: str
    T: int                  # tokens (batch * seq flattened)
    H: int                  # hidden size
    F: int                  # expert FFN inner size
    N: int                  # routed experts
    k: int                  # experts per token
    capacity_factor: float = 0.0      # <= 0: no capacity limit
    gate_bias: Optional[str] = None   # None | "zero" | "zipf1.1" | "normal"
    expert_bias: Optional[str] = None  # None | "zero" | "normal"
    sel_bias: Optional[str] = None    # None | "uniform0.1"
    F_shared: int = 0                 # 0: no shared expert
    aux_alpha: float = 0.01
    phase: str = "prefill"            # "prefill" | "decode" (which roof bounds it)
    routing: str = "token"            # "token" (top-k per token) | "expert" (top-C per expert)
    activation: str = "gelu"          # "gelu" | "silu" | "swiglu" (W1 holds gate + up rows)
    min_capacity: int = 0
    drop_order: str = "token"         # "token" | "slot"
    weight_dtype: str = "bf16"        # "bf16" | "e4m3" (FP8 codes + one fp32 scale per row)

    @property
    def w1_rows(self) -> int:
        """Rows of one expert's W1: F, or 2F (gate rows, then up rows) for SwiGLU."""
        return 2 * self.F if self.activation == "swiglu" else self.F

    def config_kwargs(self) -> dict:
        """The layer configuration of this workload, as keyword arguments of the
        binding's MoEConfig (shapes and options only)."""
        return dict(T=self.T, H=self.H, F=self.F, N=self.N, k=self.k,
                    capacity_factor=self.capacity_factor, F_shared=self.F_shared,
                    aux_alpha=self.aux_alpha, routing=self.routing, activation=self.activation,
                    min_capacity=self.min_capacity, drop_order=self.drop_order,
                    weight_dtype=self.weight_dtype)

    def with_tokens(self, T: int, name: Optional[str] = None) -> "Workload":
        return replace(self, T=T, name=name or f"{self.name}_T{T}")


# The layer shapes of the pages' models; all values synthetic.
WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    # tiny oracle case: fp32 in the source description, bf16-rounded here
    Workload("tiny", T=64, H=32, F=128, N=4, k=2, gate_bias="zero", expert_bias="zero"),
    # the pages' MoELayer: batch 8 x seq 512, hidden 1024, 8 experts, top-2, FFN 4x
    Workload("moelayer", T=4096, H=1024, F=4096, N=8, k=2, gate_bias="zero", expert_bias="zero"),
    # Mixtral-sized layer (hidden 4096, 8 experts, top-2, FFN 14336), bias-free
    Workload("mixtral_prefill", T=16384, H=4096, F=14336, N=8, k=2),
    Workload("mixtral_decode", T=64, H=4096, F=14336, N=8, k=2, phase="decode"),
    # DeepSeek-V3-sized fine-grained layer: 256 routed (top-8) + 1 shared expert
    Workload("deepseek_prefill", T=8192, H=7168, F=2048, N=256, k=8,
             sel_bias="uniform0.1", F_shared=2048),
    Workload("deepseek_decode", T=128, H=7168, F=2048, N=256, k=8,
             sel_bias="uniform0.1", F_shared=2048, phase="decode"),
    # Switch-style top-1 with capacity 1.25 and Zipf(1.1)-skewed gate offsets
    Workload("switch_capacity", T=32768, H=2048, F=8192, N=64, k=1,
             capacity_factor=1.25, gate_bias="zipf1.1"),
    # expert-choice routing on the MoELayer shapes: capacity factor 2 gives
    # each expert C = 1024 tokens, the same rows (and FLOPs) as top-2
    Workload("moelayer_expert_choice", T=4096, H=1024, F=4096, N=8, k=2, capacity_factor=2.0,
             gate_bias="zero", expert_bias="zero", routing="expert"),
    # Mixtral's gated expert: W1 holds gate and up (SwiGLU), bias-free
    Workload("mixtral_swiglu_prefill", T=16384, H=4096, F=14336, N=8, k=2, activation="swiglu"),
    Workload("mixtral_swiglu_decode", T=64, H=4096, F=14336, N=8, k=2, activation="swiglu",
             phase="decode"),
    # FP8 (E4M3) expert weights with one fp32 scale per output row: half the
    # weight bytes of the HBM-bound decode step
    Workload("mixtral_decode_fp8", T=64, H=4096, F=14336, N=8, k=2, phase="decode",
             weight_dtype="e4m3"),
    Workload("mixtral_swiglu_decode_fp8", T=64, H=4096, F=14336, N=8, k=2, activation="swiglu",
             phase="decode", weight_dtype="e4m3"),
    Workload("mixtral_prefill_fp8", T=16384, H=4096, F=14336, N=8, k=2, weight_dtype="e4m3"),
    # calibration of the expert GEMM kernel on a dense shape: one expert, so
    # the layer is two 8192 x 8192 x 8192 GEMMs (the gate is the identity)
    Workload("dense_ffn_8192", T=8192, H=8192, F=8192, N=1, k=1),
]}

# Extra small cases for tests (not benchmark lines).
TEST_WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    Workload("tiny_biased", T=64, H=32, F=128, N=4, k=2, gate_bias="normal",
             expert_bias="normal"),
    Workload("small_shared", T=300, H=256, F=384, N=16, k=4, sel_bias="uniform0.1",
             F_shared=256, expert_bias="normal"),
    Workload("small_capacity", T=1000, H=128, F=256, N=8, k=2, capacity_factor=1.0,
             gate_bias="zipf1.1"),
    Workload("small_top1", T=777, H=192, F=320, N=12, k=1, capacity_factor=1.25,
             gate_bias="zipf1.1"),
    Workload("wide_router", T=520, H=512, F=256, N=256, k=8, sel_bias="uniform0.1",
             F_shared=256),
    # ragged everything: K tails (H, F not multiples of 64), partial output
    # blocks, ragged row blocks, capacity drops, a shared expert
    Workload("odd_shapes", T=1000, H=136, F=264, N=5, k=2, capacity_factor=1.1,
             gate_bias="normal", expert_bias="normal", F_shared=72),
    Workload("dense_n1", T=300, H=64, F=96, N=1, k=1),
    Workload("all_experts", T=200, H=64, F=64, N=6, k=6, gate_bias="normal"),
    Workload("all_dropped", T=40, H=64, F=64, N=16, k=2, capacity_factor=0.1, F_shared=64),
    # more experts than the tensor-core router takes: the fp32 SIMT router runs
    Workload("many_experts", T=200, H=64, F=64, N=300, k=4, gate_bias="normal"),
    # widened rows
    Workload("small_silu", T=500, H=128, F=256, N=8, k=2, expert_bias="normal",
             activation="silu", F_shared=128),
    Workload("small_swiglu", T=600, H=192, F=320, N=8, k=2, expert_bias="normal",
             activation="swiglu", F_shared=136, gate_bias="normal"),
    Workload("swiglu_pairs", T=4096, H=256, F=384, N=4, k=2, activation="swiglu"),
    Workload("small_expert_choice", T=300, H=128, F=192, N=6, k=1, capacity_factor=1.5,
             gate_bias="normal", expert_bias="normal", routing="expert", F_shared=64),
    Workload("expert_choice_ragged", T=777, H=136, F=264, N=12, k=1, capacity_factor=0.9,
             gate_bias="zipf1.1", routing="expert", activation="swiglu"),
    Workload("expert_choice_all", T=64, H=64, F=64, N=4, k=1, capacity_factor=4.0,
             routing="expert"),
    Workload("many_experts_choice", T=200, H=64, F=64, N=300, k=1, capacity_factor=3.0,
             gate_bias="normal", routing="expert"),
    Workload("slot_major_capacity", T=1000, H=128, F=128, N=8, k=2, capacity_factor=0.8,
             gate_bias="zipf1.1", drop_order="slot"),
    Workload("min_capacity", T=40, H=64, F=64, N=16, k=2, capacity_factor=0.1, min_capacity=4,
             F_shared=64),
    Workload("small_fp8", T=300, H=256, F=384, N=8, k=2, expert_bias="normal", F_shared=256,
             weight_dtype="e4m3"),
    Workload("fp8_pairs", T=4096, H=256, F=384, N=4, k=2, weight_dtype="e4m3"),
    Workload("swiglu_fp8", T=600, H=192, F=320, N=8, k=2, activation="swiglu", F_shared=144,
             expert_bias="normal", weight_dtype="e4m3"),
    # decode-sized FP8 batches: A copies of 48 rows (T = 40) and of 16 rows
    # (capacity 6), several per A-ring slot of 128 rows
    Workload("fp8_decode_small", T=40, H=256, F=384, N=8, k=2, F_shared=128,
             expert_bias="normal", gate_bias="normal", weight_dtype="e4m3"),
    Workload("fp8_capacity_small", T=100, H=192, F=320, N=8, k=2, capacity_factor=0.5,
             activation="swiglu", gate_bias="zipf1.1", weight_dtype="e4m3"),
]}


def get_workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name in TEST_WORKLOADS:
        return TEST_WORKLOADS[name]
    raise KeyError(f"unknown workload {name!r}")


# ---------------------------------------------------------------------------
# bf16 bit helpers (data conversion only)

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def f32_to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values (|a| <= 448) to FP8 E4M3 (1 sign, 4 exponent bits
    with bias 7, 3 mantissa bits, subnormals below 2^-6) with
    round-to-nearest-even; returns the uint8 codes.  Input data generation
    only (the quantised weights are inputs of the layer)."""
    v = np.asarray(a, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    m = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint8)
    # exponent of the binade, clamped to the normal range [-6, 8]
    e = np.floor(np.log2(np.where(m > 0, m, 1.0))).astype(np.int64)
    e = np.clip(e, -6, 8)
    quantum = np.ldexp(1.0, e - 3)             # spacing of codes in this binade (2^-9 below 2^-6)
    q = np.round(m / quantum) * quantum        # numpy rounds half to even
    # rounding up can carry into the next binade: recompute its fields
    e2 = np.floor(np.log2(np.where(q > 0, q, 1.0))).astype(np.int64)
    normal = q >= 2.0 ** -6
    exp_field = np.where(normal, e2 + 7, 0)
    man_field = np.where(normal, np.round(q / np.ldexp(1.0, e2 - 3)) - 8, np.round(q / 2.0 ** -9))
    code = (exp_field << 3) | man_field.astype(np.int64)
    out[...] = np.where(q > 0, code, 0).astype(np.uint8)
    return out | sign


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# seeded draws

def _rng(seed: int, tensor: str, block: int) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(_TENSOR_ID[tensor], block))
    return np.random.Generator(np.random.PCG64(ss))


def _normal(seed, tensor, block, shape, std) -> np.ndarray:
    a = _rng(seed, tensor, block).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def gen_x_rows(w: Workload, seed: int, row0: int, row1: int) -> np.ndarray:
    """bf16 bits of activation rows [row0, row1) of x ~ N(0, 1)."""
    out = np.empty((row1 - row0, w.H), dtype=np.uint16)
    c0 = row0 // X_CHUNK_ROWS
    c1 = (row1 + X_CHUNK_ROWS - 1) // X_CHUNK_ROWS
    for c in range(c0, c1):
        lo = c * X_CHUNK_ROWS
        hi = min(lo + X_CHUNK_ROWS, w.T)
        blk = f32_to_bf16_bits(_normal(seed, "x", c, (hi - lo, w.H), 1.0))
        s0, s1 = max(lo, row0), min(hi, row1)
        out[s0 - row0:s1 - row0] = blk[s0 - lo:s1 - lo]
    return out


def gen_x(w: Workload, seed: int = 0, threads: Optional[int] = None) -> np.ndarray:
    if w.T == 0:
        return np.zeros((0, w.H), dtype=np.uint16)
    chunks = [(c * X_CHUNK_ROWS, min((c + 1) * X_CHUNK_ROWS, w.T))
              for c in range((w.T + X_CHUNK_ROWS - 1) // X_CHUNK_ROWS)]
    out = np.empty((w.T, w.H), dtype=np.uint16)

    def job(rc):
        out[rc[0]:rc[1]] = gen_x_rows(w, seed, rc[0], rc[1])
    _pool_map(job, chunks, threads)
    return out


def gen_router(w: Workload, seed: int = 0):
    """(Wg fp32 [N,H], bg fp32 [N] or None, sel_bias fp32 [N] or None)."""
    Wg = _normal(seed, "Wg", 0, (w.N, w.H), 1.0 / math.sqrt(w.H))
    bg = None
    if w.gate_bias == "zero":
        bg = np.zeros(w.N, dtype=np.float32)
    elif w.gate_bias == "zipf1.1":
        # log of a Zipf(s=1.1) pmf over experts 1..N; its normaliser is a
        # constant shift that softmax and top-k ignore, so it is dropped
        bg = (-1.1 * np.log(np.arange(1, w.N + 1, dtype=np.float64))).astype(np.float32)
    elif w.gate_bias == "normal":
        bg = _normal(seed, "bg", 0, (w.N,), 0.5)
    elif w.gate_bias is not None:
        raise ValueError(w.gate_bias)
    sel = None
    if w.sel_bias == "uniform0.1":
        sel = _rng(seed, "sel_bias", 0).uniform(-0.1, 0.1, size=w.N).astype(np.float32)
    elif w.sel_bias is not None:
        raise ValueError(w.sel_bias)
    return Wg, bg, sel


def gen_expert(w: Workload, seed: int, e: int):
    """bf16 bits of routed expert e: (W1 [F,H] ([2F,H] for SwiGLU), b1|None, W2 [H,F], b2 [H]|None)."""
    W1 = f32_to_bf16_bits(_normal(seed, "W1", e, (w.w1_rows, w.H), 1.0 / math.sqrt(w.H)))
    W2 = f32_to_bf16_bits(_normal(seed, "W2", e, (w.H, w.F), 1.0 / math.sqrt(w.F)))
    b1 = b2 = None
    if w.expert_bias == "zero":
        b1 = np.zeros(w.w1_rows, dtype=np.uint16)
        b2 = np.zeros(w.H, dtype=np.uint16)
    elif w.expert_bias == "normal":
        b1 = f32_to_bf16_bits(_normal(seed, "b1", e, (w.w1_rows,), 0.1))
        b2 = f32_to_bf16_bits(_normal(seed, "b2", e, (w.H,), 0.1))
    elif w.expert_bias is not None:
        raise ValueError(w.expert_bias)
    return W1, b1, W2, b2


def _quantise_rows(W: np.ndarray):
    """Per-row FP8: scale = max |row| / 448 (1 for an all-zero row), codes =
    E4M3(row / scale).  Returns (uint8 codes, float32 scales)."""
    amax = np.abs(W).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    return f32_to_e4m3_bits(W / scale[:, None]), scale


def gen_expert_e4m3(w: Workload, seed: int, e: int):
    """FP8 routed expert e: (W1 codes, s1, b1 bits|None, W2 codes, s2, b2 bits|None); the
    fp32 draws are those of gen_expert, then quantised per output row."""
    W1 = _normal(seed, "W1", e, (w.w1_rows, w.H), 1.0 / math.sqrt(w.H))
    W2 = _normal(seed, "W2", e, (w.H, w.F), 1.0 / math.sqrt(w.F))
    q1, s1 = _quantise_rows(W1)
    q2, s2 = _quantise_rows(W2)
    _, b1, _, b2 = gen_expert(replace(w, weight_dtype="bf16"), seed, e)
    return q1, s1, b1, q2, s2, b2


def gen_shared_e4m3(w: Workload, seed: int = 0):
    """FP8 shared expert (codes, scales, biases) or None."""
    if w.F_shared <= 0:
        return None
    Fs = w.F_shared
    Fs1 = 2 * Fs if w.activation == "swiglu" else Fs
    W1s = _normal(seed, "W1s", 0, (Fs1, w.H), 1.0 / math.sqrt(w.H))
    W2s = _normal(seed, "W2s", 0, (w.H, Fs), 1.0 / math.sqrt(Fs))
    q1, s1 = _quantise_rows(W1s)
    q2, s2 = _quantise_rows(W2s)
    sh = gen_shared(replace(w, weight_dtype="bf16"), seed)
    return q1, s1, sh[1], q2, s2, sh[3]


def gen_shared(w: Workload, seed: int = 0):
    """bf16 bits of the shared expert, or None: (W1s [Fs,H], b1s|None, W2s [H,Fs], b2s|None)."""
    if w.F_shared <= 0:
        return None
    Fs = w.F_shared
    Fs1 = 2 * Fs if w.activation == "swiglu" else Fs
    W1s = f32_to_bf16_bits(_normal(seed, "W1s", 0, (Fs1, w.H), 1.0 / math.sqrt(w.H)))
    W2s = f32_to_bf16_bits(_normal(seed, "W2s", 0, (w.H, Fs), 1.0 / math.sqrt(Fs)))
    b1s = b2s = None
    if w.expert_bias == "normal":
        b1s = f32_to_bf16_bits(_normal(seed, "b1s", 0, (Fs1,), 0.1))
        b2s = f32_to_bf16_bits(_normal(seed, "b2s", 0, (w.H,), 0.1))
    elif w.expert_bias == "zero":
        b1s = np.zeros(Fs1, dtype=np.uint16)
        b2s = np.zeros(w.H, dtype=np.uint16)
    return W1s, b1s, W2s, b2s


def gen_all(w: Workload, seed: int = 0, threads: Optional[int] = None) -> dict:
    """Every input of the layer as host arrays (bf16 tensors as uint16 bits)."""
    x = gen_x(w, seed, threads)
    Wg, bg, sel = gen_router(w, seed)
    W1 = np.empty((w.N, w.w1_rows, w.H), dtype=np.uint16)
    W2 = np.empty((w.N, w.H, w.F), dtype=np.uint16)
    has_b = w.expert_bias is not None
    b1 = np.empty((w.N, w.w1_rows), dtype=np.uint16) if has_b else None
    b2 = np.empty((w.N, w.H), dtype=np.uint16) if has_b else None

    def job(e):
        a, b, c, d = gen_expert(w, seed, e)
        W1[e] = a
        W2[e] = c
        if has_b:
            b1[e] = b
            b2[e] = d
    _pool_map(job, range(w.N), threads)
    sh = gen_shared(w, seed)
    d = dict(x=x, Wg=Wg, bg=bg, sel_bias=sel, W1=W1, b1=b1, W2=W2, b2=b2,
             W1s=None, b1s=None, W2s=None, b2s=None)
    if sh is not None:
        d.update(W1s=sh[0], b1s=sh[1], W2s=sh[2], b2s=sh[3])
    return d


def expert_getter_f64(w: Workload, seed: int = 0) -> Callable[[int], tuple]:
    """Callable e -> float64 (W1, b1, W2, b2) of routed expert e, drawn on demand."""
    cache: Dict[int, tuple] = {}

    def get(e: int):
        if e not in cache:
            W1, b1, W2, b2 = gen_expert(w, seed, e)
            cache[e] = (bf16_bits_to_f64(W1), None if b1 is None else bf16_bits_to_f64(b1),
                        bf16_bits_to_f64(W2), None if b2 is None else bf16_bits_to_f64(b2))
        return cache[e]
    return get


def shared_f64(w: Workload, seed: int = 0):
    sh = gen_shared(w, seed)
    if sh is None:
        return None
    return tuple(None if a is None else bf16_bits_to_f64(a) for a in sh)


def _pool_map(fn, items, threads):
    items = list(items)
    n = threads or min(len(items), os.cpu_count() or 1, 64)
    if n <= 1 or len(items) <= 1:
        for it in items:
            fn(it)
        return
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(fn, items))


# ---------------------------------------------------------------------------
# device upload (data movement only; torch is imported lazily)

def bits_to_torch_bf16(a: np.ndarray, device="cpu"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


# names of the layer parameters (the fields of the binding's MoEWeights)
WEIGHT_KEYS = ("Wg", "bg", "sel_bias", "W1", "b1", "W2", "b2", "W1s", "b1s", "W2s", "b2s",
               "s1", "s2", "s1s", "s2s")


def same_weights(a: Workload, b: Workload) -> bool:
    """True when the two workloads draw identical layer parameters (they
    differ at most in the token count and the routing options)."""
    return (a.H, a.F, a.N, a.F_shared, a.activation, a.weight_dtype, a.expert_bias, a.gate_bias,
            a.sel_bias) == (b.H, b.F, b.N, b.F_shared, b.activation, b.weight_dtype,
                            b.expert_bias, b.gate_bias, b.sel_bias)


def to_device(w: Workload, seed: int = 0, device="cuda", x_seed: Optional[int] = None,
              reuse: Optional[dict] = None) -> dict:
    """Draws every input on the host (per-expert blocks in threads) and copies
    it to `device`.  Returns a dict of torch tensors with the layer's names
    (WEIGHT_KEYS, None where absent) plus ``x`` and ``x_bits`` (the host bf16
    bits of x).  FP8 workloads hold uint8 E4M3 codes in W1, W2, W1s, W2s and
    their fp32 row scales in s1, s2, s1s, s2s.  ``reuse``: the result of an
    earlier call for a workload with the same parameters (same_weights); its
    weight tensors are shared and only x is drawn."""
    import torch
    fp8 = w.weight_dtype == "e4m3"
    x_bits = gen_x(w, seed if x_seed is None else x_seed)
    if reuse is not None:
        d = {k: reuse[k] for k in WEIGHT_KEYS}
        d.update(x_bits=x_bits, x=bits_to_torch_bf16(x_bits, device))
        return d
    Wg, bg, sel = gen_router(w, seed)
    wdt = torch.uint8 if fp8 else torch.bfloat16
    W1 = torch.empty((w.N, w.w1_rows, w.H), dtype=wdt, device=device)
    W2 = torch.empty((w.N, w.H, w.F), dtype=wdt, device=device)
    s1 = torch.empty((w.N, w.w1_rows), dtype=torch.float32, device=device) if fp8 else None
    s2 = torch.empty((w.N, w.H), dtype=torch.float32, device=device) if fp8 else None
    has_b = w.expert_bias is not None
    b1 = torch.empty((w.N, w.w1_rows), dtype=torch.bfloat16, device=device) if has_b else None
    b2 = torch.empty((w.N, w.H), dtype=torch.bfloat16, device=device) if has_b else None
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    bf = lambda a: None if a is None else bits_to_torch_bf16(a, device)
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint8))
    batch = 32
    gen = (lambda e: gen_expert_e4m3(w, seed, e)) if fp8 else (lambda e: gen_expert(w, seed, e))
    with ThreadPoolExecutor(min(32, max(1, w.N))) as ex:
        for e0 in range(0, w.N, batch):
            blocks = ex.map(gen, range(e0, min(w.N, e0 + batch)))
            for j, blk in enumerate(blocks):
                e = e0 + j
                if fp8:
                    q1, sc1, b, q2, sc2, d = blk
                    W1[e].copy_(u8(q1))
                    W2[e].copy_(u8(q2))
                    s1[e].copy_(torch.from_numpy(sc1))
                    s2[e].copy_(torch.from_numpy(sc2))
                else:
                    a, b, c, d = blk
                    W1[e].copy_(bits_to_torch_bf16(a))
                    W2[e].copy_(bits_to_torch_bf16(c))
                if has_b:
                    b1[e].copy_(bits_to_torch_bf16(b))
                    b2[e].copy_(bits_to_torch_bf16(d))
    d = dict(x_bits=x_bits, x=bits_to_torch_bf16(x_bits, device), Wg=f32(Wg), bg=f32(bg),
             sel_bias=f32(sel), W1=W1, b1=b1, W2=W2, b2=b2, W1s=None, b1s=None, W2s=None, b2s=None,
             s1=s1, s2=s2, s1s=None, s2s=None)
    if fp8:
        sh = gen_shared_e4m3(w, seed)
        if sh is not None:
            d.update(W1s=u8(sh[0]).to(device), s1s=f32(sh[1]), b1s=bf(sh[2]),
                     W2s=u8(sh[3]).to(device), s2s=f32(sh[4]), b2s=bf(sh[5]))
    else:
        sh = gen_shared(w, seed)
        if sh is not None:
            d.update(W1s=bf(sh[0]), b1s=bf(sh[1]), W2s=bf(sh[2]), b2s=bf(sh[3]))
    return d
