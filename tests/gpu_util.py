"""Helpers for the GPU parity tests: tolerances and comparisons (no attention math)."""
import math

import numpy as np
import torch

# Tolerances stated for the hot path: fp32 inputs max-abs 1e-4 on O and 1e-5 on
# LSE; bf16 inputs (fp32 accumulation) max-abs 2e-2 and mean-abs 2e-3 on O and
# 1e-2 on LSE.
F32_O, F32_LSE = 1e-4, 1e-5
BF16_O_MAX, BF16_O_MEAN, BF16_LSE = 2e-2, 2e-3, 1e-2


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(got, want, dtype):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - want)
    if dtype == "f32":
        assert err.max() <= F32_O, f"max-abs {err.max():.3e}"
    else:
        assert err.max() <= BF16_O_MAX, f"max-abs {err.max():.3e}"
        assert err.mean() <= BF16_O_MEAN, f"mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def check_lse(got, want, dtype):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    ninf_g, ninf_w = np.isneginf(got), np.isneginf(want)
    assert (ninf_g == ninf_w).all(), "empty-row pattern differs"
    fin = ~ninf_w
    if fin.any():
        err = np.abs(got[fin] - want[fin]).max()
        assert err <= (F32_LSE if dtype == "f32" else BF16_LSE), f"lse max-abs {err:.3e}"
        return float(err)
    return 0.0
