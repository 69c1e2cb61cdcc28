"""The log-domain evaluation of the forward pass (csa_forward_logdomain:
z = a + b with b from log phi2 of the logit steps, eq. (10)/(11) as
written) against the oracle, at the forward pass's bars, and against the
interval-share kernel csa_forward on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import forward
from continuous_softmax_attention_gb300.inputs import make_inputs, workload_inputs
from gpu_util import assert_close, boundary_rows, np64, to_dev

pytestmark = pytest.mark.gpu


def run(x, scale, mode, log_domain=True):
    g = to_dev(x)
    o, lse = forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale,
                     log_domain=log_domain)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("d", [64, 128, 96])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("T", [1, 2, 109, 110, 111, 126, 127, 128, 221, 300, 700])
def test_logdomain_bf16(d, mode, T):
    x = make_inputs(1, 2, T, d, "bf16", seed=610 + T + d + mode)
    scale = 1.0 / d ** 0.5
    o, lse = run(x, scale, mode)
    ro, rl = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    assert_close(o, lse, ro, rl, "bf16", f"log-domain d={d} mode={mode} T={T}")


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0, -0.1, -1.0])
@pytest.mark.parametrize("mode", [0, 1])
def test_logdomain_logit_ranges(scale, mode):
    # scale 4 at d = 64: logit steps of order +-100 (log phi2 on its
    # large-|x| branches, the running max raised); negative scales too
    x = make_inputs(2, 4, 512, 64, "bf16", seed=620)
    o, lse = run(x, scale, mode)
    ro, rl = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    assert_close(o, lse, ro, rl, "bf16", f"scale={scale} mode={mode}")


def test_logdomain_matches_interval_kernel():
    # the two evaluations of the same weights on the same inputs: their
    # outputs differ by the bf16 rounding of the weights at most
    x = make_inputs(2, 4, 1000, 128, "bf16", seed=630)
    o1, l1 = run(x, 1.0 / 128 ** 0.5, 0, log_domain=True)
    o2, l2 = run(x, 1.0 / 128 ** 0.5, 0, log_domain=False)
    assert np.abs(np64(o1) - np64(o2)).max() <= 2e-2
    assert np.abs(np64(l1) - np64(l2)).max() <= 1e-3


def test_logdomain_mid_sampled():
    x = workload_inputs("mid")
    B, H, T, d = x["q"].shape
    scale = 1.0 / d ** 0.5
    o, lse = run(x, scale, 0)
    rows = boundary_rows(T, extra=list(range(0, T, 331)))
    picks = [(b, h, r) for b in (0, B - 1) for h in (0, H - 1) for r in rows]
    flat = oracle.flat_rows(B, H, T, picks)
    ro, rl = oracle.forward_rows(x["q"], x["k"], x["v"], flat, scale=scale)
    go = o.reshape(-1, d)[torch.as_tensor(flat)]
    gl = lse.reshape(-1)[torch.as_tensor(flat)]
    assert_close(go, gl, ro, rl, "bf16", "mid rows")


def test_logdomain_rejects_fp32_and_two_forms():
    x = make_inputs(1, 1, 8, 16, "f32", seed=640)
    g = to_dev(x)
    with pytest.raises(ValueError):
        forward(g["q"], g["k"], g["v"], log_domain=True)
    y = to_dev(make_inputs(1, 1, 8, 64, "bf16", seed=641))
    with pytest.raises(ValueError):
        forward(y["q"], y["k"], y["v"], log_domain=True, short_conv=True)
