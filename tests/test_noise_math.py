"""Host checks of the arithmetic behind the device's fast E = -ln u (no GPU).

Below t = 1 - u = 1/8 the kernels evaluate -ln(1 - t) by its Taylor series to
t^8 / 8 in Horner form; this emulates that evaluation in fp32 on the uniform
grid u = (n + 0.5) 2^-23 and compares it with fp64 log1p.
"""

import numpy as np


def _series_f32(t):
    t = t.astype(np.float32)
    s = np.float32(0.125) * t + np.float32(0.142857142857)
    for c in (0.166666666667, 0.2, 0.25, 0.333333333333, 0.5, 1.0):
        s = s * t + np.float32(c)
    return s * t


def test_series_branch_is_accurate_on_the_uniform_grid():
    # every grid point with t < 1/8 near the top (the fast arrivals), plus a sample
    n_top = np.arange(0, 1 << 16)
    n_mid = np.random.default_rng(0).integers(0, 1 << 20, 200_000)
    t = ((np.concatenate([n_top, n_mid]) + 0.5) * 2.0 ** -23)
    t = t[t < 0.125]
    approx = _series_f32(t).astype(np.float64)
    exact = -np.log1p(-t)
    rel = np.abs(approx - exact) / exact
    assert rel.max() < 3e-7
