"""The FP8 weight inputs: the generator's E4M3 rounding agrees with torch's
float8_e4m3fn conversion (round to nearest even), and the per-row scales put
each row's largest magnitude on the largest code."""
import numpy as np
import torch

import moe_workloads as wl
from oracle import moe_oracle as O


def test_e4m3_encoder_matches_torch():
    rng = np.random.default_rng(3)
    v = np.clip(rng.standard_normal(100000).astype(np.float32) * 60, -448, 448)
    edge = np.array([0.0, -0.0, 2 ** -10, 3 * 2 ** -10, 2 ** -9, 1.0625, 1.1875, 448, -448,
                     2 ** -6, 2 ** -6 * 1.0625, 15.5, 232.0, -0.00048828125], dtype=np.float32)
    v = np.concatenate([v, edge])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(wl.f32_to_e4m3_bits(v), ref)


def test_rows_are_scaled_to_the_largest_code():
    w = wl.get_workload("small_fp8")
    q1, s1, b1, q2, s2, b2 = wl.gen_expert_e4m3(w, 0, 3)
    assert q1.dtype == np.uint8 and q1.shape == (w.F, w.H) and s1.shape == (w.F,)
    assert q2.shape == (w.H, w.F) and s2.shape == (w.H,)
    W = O.dequantize_rows(q1, s1)
    assert np.allclose(np.abs(W).max(axis=1), 448.0 * s1)
    # the quantised rows stay within half a code step of the fp32 draws
    W1f = wl._normal(0, "W1", 3, (w.F, w.H), 1.0 / np.sqrt(w.H))
    assert np.all(np.abs(W - W1f) <= np.abs(W1f) * 2.0 ** -4 + s1[:, None] * 2.0 ** -10)
