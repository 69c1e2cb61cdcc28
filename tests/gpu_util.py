"""Helpers shared by the GPU tests: device copies and the parity bars.

Tolerances (the method's acceptance bars):
  fp32 inputs : max |o - oracle| <= 1e-5 and max |lse - oracle| <= 1e-5
  bf16 inputs : max |o - oracle| <= 2e-2, mean |o - oracle| <= 2e-3,
                max |lse - oracle| <= 1e-3
The oracle is fed exactly the values the GPU sees (bf16-rounded for bf16).
"""
import numpy as np
import torch

F32_TOL = 1e-5
BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


def to_dev(x, dev="cuda"):
    return {k: v.to(dev) for k, v in x.items()}


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(o, lse, ro, rl, dtype, what=""):
    o = np64(o) if torch.is_tensor(o) else o
    lse = np64(lse) if torch.is_tensor(lse) else lse
    err = np.abs(o - ro)
    lerr = np.abs(lse - rl)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    if dtype == "f32":
        assert err.max() <= F32_TOL, f"{what}: max |o err| {err.max():.3g}"
        assert lerr.max() <= F32_TOL, f"{what}: max |lse err| {lerr.max():.3g}"
    else:
        assert err.max() <= BF16_MAX, f"{what}: max |o err| {err.max():.3g}"
        assert err.mean() <= BF16_MEAN, f"{what}: mean |o err| {err.mean():.3g}"
        assert lerr.max() <= LSE_TOL, f"{what}: max |lse err| {lerr.max():.3g}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def boundary_rows(T, extra=()):
    """Rows around every tile edge of the kernels: query tiles of 128 rows
    (pairs of 256), key tiles every 110 (d = 128) or 126 (d = 64) keys, and
    the 128-key tiles of the standard kernel."""
    rows = set(extra)
    for base in (110, 126, 128, 256):
        n = 1
        while base * n - 2 < T:
            for dlt in (-2, -1, 0, 1):
                r = base * n + dlt
                if 0 <= r < T:
                    rows.add(r)
            n += 1
    rows.update(r for r in (0, 1, 2, T - 2, T - 1) if 0 <= r < T)
    return sorted(rows)
