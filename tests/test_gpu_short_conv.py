"""The short-conv reading of eq. (13) (csa_forward_short_conv and _f32)
against the oracle's forward_short_conv, at the forward pass's bars."""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import forward
from continuous_softmax_attention_gb300.inputs import make_inputs, workload_inputs
from gpu_util import assert_close, boundary_rows, to_dev

pytestmark = pytest.mark.gpu


def run(x, scale, mode):
    g = to_dev(x)
    o, lse = forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale,
                     short_conv=True)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_short_conv_f32(mode):
    x = make_inputs(2, 3, 67, 24, "f32", seed=200 + mode)
    o, lse = run(x, 0.4, mode)
    ro, rl = oracle.forward_short_conv(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.4, mode=mode)
    assert_close(o, lse, ro, rl, "f32", f"f32 mode={mode}")


@pytest.mark.parametrize("d", [64, 128, 96])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("T", [1, 2, 109, 110, 111, 127, 128, 221, 300, 700])
def test_short_conv_bf16(d, mode, T):
    x = make_inputs(1, 2, T, d, "bf16", seed=210 + T + d + mode)
    scale = 1.0 / d ** 0.5
    o, lse = run(x, scale, mode)
    ro, rl = oracle.forward_short_conv(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale,
                                       mode=mode)
    assert_close(o, lse, ro, rl, "bf16", f"bf16 d={d} mode={mode} T={T}")


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0])
def test_short_conv_logit_ranges(scale):
    # scale 4 at d = 64: logit steps of order +-100; the first-order form
    # stays a softmax of bounded arguments
    x = make_inputs(2, 2, 300, 64, "bf16", seed=220)
    o, lse = run(x, scale, 0)
    ro, rl = oracle.forward_short_conv(x["q"], x["k"], x["v"], scale=scale)
    assert_close(o, lse, ro, rl, "bf16", f"scale={scale}")


def test_short_conv_headline_sampled():
    x = workload_inputs("headline")
    B, H, T, d = x["q"].shape
    o, lse = run(x, 1.0 / d ** 0.5, 0)
    rows = boundary_rows(T, extra=list(range(0, T, 997)))
    picks = [(0, h, r) for h in (0, H - 1) for r in rows]
    flat = oracle.flat_rows(B, H, T, picks)
    ro, rl = oracle.forward_short_conv_rows(x["q"], x["k"], x["v"], flat, scale=1.0 / d ** 0.5)
    go = o.reshape(-1, d)[torch.as_tensor(flat)]
    gl = lse.reshape(-1)[torch.as_tensor(flat)]
    assert_close(go, gl, ro, rl, "bf16", "headline rows")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_short_conv_running_max_raised(d, mode):
    """Keys far into the sequence whose logits exceed every earlier one by
    hundreds (log2 units): the running max is raised (at d = 128 by both
    column halves together, as they share one accumulator) and what was
    written rescaled.  The oracle is exact for any logits."""
    T = 700
    x = make_inputs(1, 2, T, d, "bf16", seed=230 + d)
    k = x["k"].float()
    for pos, f in ((300, 25.0), (301, 25.0), (450, 60.0), (640, 90.0)):
        k[:, :, pos] = k[:, :, pos] * f
    x["k"] = k.to(torch.bfloat16)
    scale = 1.0 / d ** 0.5
    o, lse = run(x, scale, mode)
    ro, rl = oracle.forward_short_conv(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale,
                                       mode=mode)
    assert_close(o, lse, ro, rl, "bf16", f"short conv, max raised d={d} mode={mode}")
