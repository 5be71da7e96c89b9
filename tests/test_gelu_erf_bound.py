"""The expert GELU's erf is Abramowitz & Stegun, "Handbook of Mathematical
Functions", formula 7.1.26 (|error| <= 1.5e-7).  This CPU test evaluates that
published formula in float32, the precision the kernel uses, and checks its
error against float64 erf over the range GELU sees; the GPU parity tests then
check the whole GEMM1 + GELU output against the oracle's exact erf."""
import numpy as np
from scipy.special import erf

# A&S 7.1.26 coefficients (Handbook of Mathematical Functions, table of 7.1.26)
P = 0.3275911
A = [0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429]


def erf_as7126_f32(x):
    x = np.asarray(x, np.float32)
    ax = np.abs(x)
    t = np.float32(1.0) / (np.float32(P) * ax + np.float32(1.0))
    poly = np.float32(A[4])
    for a in A[3::-1]:
        poly = poly * t + np.float32(a)
    poly = poly * t
    r = np.float32(1.0) - poly * np.exp(-ax * ax).astype(np.float32)
    return np.copysign(r, x)


def test_erf_bound_float32():
    x = np.linspace(-8, 8, 400001).astype(np.float32)
    err = np.abs(erf_as7126_f32(x).astype(np.float64) - erf(x.astype(np.float64)))
    assert err.max() < 1.5e-7 + 4e-7   # the formula's bound plus float32 evaluation


def test_gelu_error_far_below_bf16_rounding():
    z = np.linspace(-10, 10, 200001).astype(np.float32)
    g = 0.5 * z * (1 + erf_as7126_f32(z / np.sqrt(np.float32(2))))
    g_ref = 0.5 * z.astype(np.float64) * (1 + erf(z.astype(np.float64) / np.sqrt(2)))
    # bf16 keeps 8 significant bits: half an ulp is 2^-9 relative
    assert (np.abs(g - g_ref) <= 1e-6 * np.maximum(1.0, np.abs(z))).all()
