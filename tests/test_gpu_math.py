"""GPU checks of the library's device math and its bounded waits."""
import math

import numpy as np
import pytest
import torch

import continuous_softmax_attention_gb300 as csa
import oracle

pytestmark = pytest.mark.gpu


def test_logphi2_device_function():
    """The fp32 log phi2 of the CUDA-core kernels against the oracle's double
    log phi2, over x in [-1000, 1000] (eq. (6))."""
    xs = np.concatenate([
        np.linspace(-1000, 1000, 20001),
        np.linspace(-1.5, 1.5, 3001),
        np.array([0.0, 1e-30, -1e-30, 1e-8, -1e-8, 1.0, -1.0, np.nextafter(1.0, 2), -np.nextafter(1.0, 2)]),
    ]).astype(np.float32)
    y = csa.logphi2_eval(torch.from_numpy(xs).cuda()).cpu().numpy().astype(np.float64)
    ref = np.array([oracle.log_phi2(float(x)) for x in xs])
    err = np.abs(y - ref) / np.maximum(1.0, np.abs(ref))
    assert np.isfinite(y).all()
    assert err.max() < 2e-6, (err.max(), xs[err.argmax()])


def test_segment_weights_against_phi2():
    """The tensor-core kernel's interval weights R = p0 phi2(x), L = p1 phi2(-x)
    (the regrouping of eq. (9)) against the oracle's phi2, over steps x from
    0 to +-300 and levels u <= 0."""
    rng = np.random.default_rng(0)
    x = np.concatenate([np.zeros(16), rng.uniform(-1, 1, 4000) * 10.0 ** rng.uniform(-7, 0, 4000),
                        rng.uniform(-12, 12, 4000), rng.uniform(-300, 300, 2000)])
    u0 = -rng.uniform(0, 30, x.size)
    u1 = u0 + x
    top = np.maximum(u0, u1)
    u0, u1 = u0 - top, u1 - top  # max(u0, u1) = 0 as after the running max
    u0 = u0.astype(np.float32)
    u1 = u1.astype(np.float32)
    r, l_ = csa.segment_weights_eval(torch.from_numpy(u0).cuda(), torch.from_numpy(u1).cuda())
    r = r.cpu().numpy().astype(np.float64)
    l_ = l_.cpu().numpy().astype(np.float64)
    xx = u1.astype(np.float64) - u0.astype(np.float64)
    p0, p1 = np.exp(u0.astype(np.float64)), np.exp(u1.astype(np.float64))
    rr = np.array([a * oracle.phi2(s) for a, s in zip(p0, xx)])
    rl = np.array([b * oracle.phi2(-s) for b, s in zip(p1, xx)])
    # Bound: the kernel's closed form loses ~1.4e-6/X^2 (X in log2 units) to the
    # rounding of the two exponentials, and below |X| = 1/16 it switches to a
    # first-order series with error (ln2 X)^2/12; both stay under 4e-4
    # relative, below the 2^-9 rounding of the bf16 P these weights become.
    assert np.isfinite(r).all() and np.isfinite(l_).all()
    assert np.abs(r - rr).max() < 3e-4, np.abs(r - rr).max()
    assert np.abs(l_ - rl).max() < 3e-4, np.abs(l_ - rl).max()
    big = rr > 1e-3
    assert (np.abs(r - rr)[big] / rr[big]).max() < 1e-3


def test_bounded_wait_times_out_without_fault():
    """A wait on an mbarrier that nothing completes gives up, records the
    timeout status, and leaves the context usable."""
    assert csa.device_status() == 0
    csa.selftest_wait_timeout(2000)
    torch.cuda.synchronize()
    assert csa.device_status() == csa._lib.CSA_ERR_TIMEOUT
    assert csa.device_status() == 0  # read clears it
    x = torch.randn(1, 1, 8, 64, device="cuda", dtype=torch.bfloat16)
    o, _ = csa.forward(x, x, x)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert csa.device_status() == 0
