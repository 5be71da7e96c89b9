"""Every E4M3 weight code through the FP8 expert FFN, compared value by value.

One expert (F = H = 256, scale 1, no biases, SiLU) whose second Linear is the
identity and whose input rows are one-hot: row t of the first Linear's output
is then column t of W1 decoded, and the layer returns SiLU of each decoded
weight, rounded to bf16 once in the hidden layer (the identity Linear and the
weight 1 add no rounding).  Column t of W1 holds every code except the two NaN
codes, so the widening of each code to bf16 (signs, zeros, the subnormal
codes m * 2^-9, the largest normal 448) is checked to within one bf16 step of
the oracle's SiLU (SiLU keeps its relative accuracy for negative inputs,
where GELU's 1 + erf cancels).  A subnormal flushed to zero, a dropped sign
or an exponent off by one fails by far more.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

H = F = 256
NAN_CODES = (0x7F, 0xFF)


def _codes():
    i = np.arange(F)[:, None]
    t = np.arange(H)[None, :]
    c = ((i + 7 * t) % 256).astype(np.uint8)     # W1[i, t]: a permutation of 0..255 per column
    c[np.isin(c, NAN_CODES)] = 0
    return c


def test_every_code_widens_exactly():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_72_b300 as m
    T = H
    cfg = m.MoEConfig(T=T, H=H, F=F, N=1, k=1, activation="silu", weight_dtype="e4m3")
    W1c = _codes()
    W2c = np.zeros((H, F), np.uint8)
    np.fill_diagonal(W2c, 0x38)                   # E4M3 1.0
    dev = "cuda"
    weights = m.MoEWeights(
        Wg=torch.zeros((1, H), dtype=torch.float32, device=dev),
        W1=torch.from_numpy(W1c[None]).to(dev), W2=torch.from_numpy(W2c[None]).to(dev),
        s1=torch.ones((1, F), dtype=torch.float32, device=dev),
        s2=torch.ones((1, H), dtype=torch.float32, device=dev))
    x = torch.eye(T, H, dtype=torch.bfloat16, device=dev)   # token t = one-hot at t
    perm = torch.arange(T, dtype=torch.int32, device=dev)
    offsets = torch.tensor([0, T], dtype=torch.int32, device=dev)
    topk_w = torch.ones((T, 1), dtype=torch.float32, device=dev)
    y, _ = m.moe_expert_ffn(cfg, x, perm, offsets, topk_w, weights)
    torch.cuda.synchronize()
    got = y[:T].float().cpu().numpy().astype(np.float64)

    # row t, column i: SiLU(decode(W1[i, t])), the hidden value rounded to bf16
    v = O.e4m3_decode(W1c.T)                      # [t, i]
    want = O.silu(v)
    assert np.isfinite(want).all()
    # the decoded codes themselves span the format's special values
    flat = v.ravel()
    assert (flat == 448.0).any() and (flat == -448.0).any()
    assert (flat == 2.0 ** -9).any() and (flat == 7 * 2.0 ** -9).any()
    assert np.signbit(flat[flat == 0]).any()      # -0 (code 0x80) is present
    tol = 2.0 ** -7 * np.abs(want) + 1e-30        # one bf16 step, with margin
    err = np.abs(got - want)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (
        f"{len(bad)} mismatches, e.g. code {W1c[bad[0][1], bad[0][0]]:#04x}: "
        f"got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}")
    # every nonzero subnormal code gives a nonzero output
    sub = np.abs(v) < 2.0 ** -6
    assert np.all(got[sub & (v != 0)] != 0)
