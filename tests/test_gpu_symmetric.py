"""The symmetric interval [1/2, t + 1/2] (csa_forward_symmetric and _f32)
against the oracle's forward_symmetric, at the forward pass's bars."""
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import forward_symmetric
from continuous_softmax_attention_gb300.inputs import make_inputs, workload_inputs
from gpu_util import assert_close, boundary_rows, to_dev

pytestmark = pytest.mark.gpu


def run(x, scale):
    g = to_dev(x)
    o, lse = forward_symmetric(g["q"], g["k"], g["v"], scale=scale)
    torch.cuda.synchronize()
    return o, lse


def test_symmetric_f32():
    x = make_inputs(2, 3, 67, 24, "f32", seed=300)
    o, lse = run(x, 0.4)
    ro, rl = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=0.4)
    assert_close(o, lse, ro, rl, "f32", "f32")


@pytest.mark.parametrize("d", [64, 128, 96])
@pytest.mark.parametrize("T", [1, 2, 3, 109, 110, 111, 126, 127, 128, 129, 220, 254, 255, 300, 700])
def test_symmetric_bf16(d, T):
    x = make_inputs(1, 2, T, d, "bf16", seed=310 + T + d)
    scale = 1.0 / d ** 0.5
    o, lse = run(x, scale)
    ro, rl = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=scale)
    assert_close(o, lse, ro, rl, "bf16", f"bf16 d={d} T={T}")


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0])
def test_symmetric_logit_ranges(scale):
    # scale 4 at d = 64: logit steps of order +-100, and every sink-free row
    # must still be normalised by its own keys
    x = make_inputs(2, 2, 300, 64, "bf16", seed=320)
    o, lse = run(x, scale)
    ro, rl = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=scale)
    assert_close(o, lse, ro, rl, "bf16", f"scale={scale}")


def test_symmetric_headline_sampled():
    x = workload_inputs("headline")
    B, H, T, d = x["q"].shape
    o, lse = run(x, 1.0 / d ** 0.5)
    rows = boundary_rows(T, extra=list(range(0, T, 997)))
    picks = [(0, h, r) for h in (0, H - 1) for r in rows]
    flat = oracle.flat_rows(B, H, T, picks)
    ro, rl = oracle.forward_symmetric_rows(x["q"], x["k"], x["v"], flat, scale=1.0 / d ** 0.5)
    idx = torch.as_tensor(flat)
    assert_close(o.reshape(-1, d)[idx], lse.reshape(-1)[idx], ro, rl, "bf16", "headline rows")
