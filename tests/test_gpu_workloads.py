"""The method's evaluation workloads at full size, in the launch configuration
the benchmark times, checked against the oracle: whole heads where the
oracle is quick, and otherwise rows sampled at every tile edge plus random
rows of every head (the oracle computes those one by one)."""
import math

import numpy as np
import pytest
import torch

import continuous_softmax_attention_gb300 as csa
import oracle
from continuous_softmax_attention_gb300.inputs import WORKLOADS, workload_inputs
from gpu_util import assert_close, boundary_rows, np64, to_dev

pytestmark = pytest.mark.gpu


def _sampled(x, o, lse, mode, scale, rows_per_head, std=False, seed=0):
    B, H, T, d = x["q"].shape
    rng = np.random.default_rng(seed)
    picks = []
    edges = boundary_rows(T)
    for b in range(B):
        for h in range(H):
            chosen = set(rng.choice(edges, size=min(len(edges), rows_per_head), replace=False).tolist())
            chosen.update(rng.integers(0, T, size=4).tolist())
            picks += [(b, h, int(r)) for r in sorted(chosen)]
    rows = oracle.flat_rows(B, H, T, picks)
    ro, rl = oracle.forward_rows(x["q"], x["k"], x["v"], rows, x["k0"], x["v0"], scale=scale,
                                 mode=mode, std=std)
    og = np64(o).reshape(-1, d)[rows]
    lg = np64(lse).reshape(-1)[rows]
    return assert_close(og, lg, ro, rl, "bf16", "sampled rows")


def _full_heads(x, o, lse, mode, scale, heads, std=False):
    """Every row of the given heads (the oracle's row form, which spreads the
    rows over the host's cores)."""
    B, H, T, d = x["q"].shape
    for (b, h) in heads:
        rows = oracle.flat_rows(B, H, T, [(b, h, r) for r in range(T)])
        ro, rl = oracle.forward_rows(x["q"], x["k"], x["v"], rows, x["k0"], x["v0"], scale=scale,
                                     mode=mode, std=std)
        og = np64(o).reshape(-1, d)[rows]
        lg = np64(lse).reshape(-1)[rows]
        assert_close(og, lg, ro, rl, "bf16", f"head {b},{h}")


def _run(name):
    w = WORKLOADS[name]
    x = workload_inputs(name)
    g = to_dev(x)
    scale = 1.0 / math.sqrt(w.d)
    mode = w.modes[0]
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    return w, x, g, o, lse, mode, scale


def test_mid_workload():
    """B=4, H=16, T=2048, d=128, RoPE on q and k, zero sink."""
    w, x, g, o, lse, mode, scale = _run("mid")
    _full_heads(x, o, lse, mode, scale, [(0, 0), (3, 15)])
    _sampled(x, o, lse, mode, scale, rows_per_head=12, seed=1)


def test_headline_workload():
    """B=1, H=32, T=8192, d=128, zero sink; and the standard kernel on it.
    Every row of two heads (one in each scheduling group of 16 heads), tile
    edges and random rows of all the others."""
    w, x, g, o, lse, mode, scale = _run("headline")
    _full_heads(x, o, lse, mode, scale, [(0, 0), (0, 31)])
    _sampled(x, o, lse, mode, scale, rows_per_head=8, seed=2)
    so, sl = csa.std_forward(g["q"], g["k"], g["v"], scale=scale)
    torch.cuda.synchronize()
    _sampled(x, so, sl, mode, scale, rows_per_head=6, std=True, seed=3)


def test_long_workload():
    """B=1, H=8, T=32768, d=64, given per-head k0, v0 (trainable-sink mode).
    Every row of the first and last heads (about 20 s of oracle work each),
    tile edges and random rows of all heads."""
    w, x, g, o, lse, mode, scale = _run("long")
    _full_heads(x, o, lse, mode, scale, [(0, 0), (0, 7)])
    _sampled(x, o, lse, mode, scale, rows_per_head=24, seed=4)


def test_forward_very_long_rows():
    """T = 131072 (1024 query tiles, 1033 key tiles per head): index and TMA
    coordinate arithmetic at length, checked on the last rows and every few
    thousandth row against the oracle."""
    B, H, T, d = 1, 2, 131072, 64
    from continuous_softmax_attention_gb300.inputs import make_inputs

    x = make_inputs(B, H, T, d, "bf16", seed=500)
    g = to_dev(x)
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=2)
    torch.cuda.synchronize()
    rows = sorted(set([0, 1, 126, 127, 128, T - 129, T - 2, T - 1] + list(range(0, T, 9973))))
    picks = [(0, h, r) for h in range(H) for r in rows]
    flat = oracle.flat_rows(B, H, T, picks)
    ro, rl = oracle.forward_rows(x["q"], x["k"], x["v"], flat, x["k0"], x["v0"],
                                 scale=1.0 / d ** 0.5, mode=2)
    idx = torch.as_tensor(flat)
    assert_close(o.reshape(-1, d)[idx], lse.reshape(-1)[idx], ro, rl, "bf16", "T=131072")
