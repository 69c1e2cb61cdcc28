"""Pins of the backward oracle (oracle.backward, csa_oracle_backward.c).

Nothing here re-types the oracle's chain rule.  The gradients are checked
against:
  * central finite differences of the eq. (8) forward oracle (a different
    closed form of the same forward pass) on L = sum(dout * o);
  * torch autograd through a float64 transcription of eq. (10)/(11);
  * invariants of the method: translating every key (the sink included) by
    one vector leaves o unchanged, translating every value by c moves o by
    c, and with scale = 0 the weights do not depend on q or k;
  * phi2'(x) against 50-digit numerical integration of its integral form.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300.inputs import make_inputs

MODES = (oracle.ZERO, oracle.COPY_FIRST, oracle.GIVEN)


def test_log_dphi2_against_integral():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    for x in (0.0, 1e-9, -1e-9, 0.3, -0.3, 0.4999999, 0.5, -0.5, -0.5000001, 1.0, -1.0, 2.0,
              -2.0, 7.5, -7.5, 40.0, -40.0, 300.0, -300.0):
        xm = mpmath.mpf(x)
        ref = mpmath.log(mpmath.quad(lambda s: s * (1 - s) * mpmath.exp(s * xm), [0, 0.5, 1]))
        got = oracle.log_dphi2(x)
        assert abs(got - float(ref)) <= 1e-13 * max(1.0, abs(float(ref))), (x, got, float(ref))


def _loss(x, g, scale, mode):
    o, _ = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode,
                          nthreads=1)
    return float((o * g.numpy().astype(np.float64)).sum())


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("scale", [0.4, 1.7])
def test_backward_matches_finite_differences(mode, scale):
    x = make_inputs(1, 2, 5, 3, "f32", seed=11 + mode)
    g = torch.randn(1, 2, 5, 3, generator=torch.Generator().manual_seed(5))
    ref = oracle.backward(x["q"], x["k"], x["v"], g, x["k0"], x["v0"], scale=scale, mode=mode)
    h = 2.0 ** -10
    names = ["q", "k", "v"] + (["k0", "v0"] if mode == oracle.GIVEN else [])
    for name in names:
        t = x[name]
        fd = np.zeros(t.shape, dtype=np.float64)
        for idx in np.ndindex(*t.shape):
            orig = float(t[idx])
            t[idx] = orig + h
            lp = _loss(x, g, scale, mode)
            t[idx] = orig - h
            lm = _loss(x, g, scale, mode)
            t[idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        got = ref["d" + name]
        err = np.abs(got - fd).max()
        assert err <= 2e-6 * max(1.0, np.abs(fd).max()), (name, err)


def _torch_forward(q, k, v, k0, v0, scale, mode):
    """eq. (10)/(11) in float64 torch ops, one row at a time."""
    B, H, T, d = q.shape
    outs = []
    for b in range(B):
        for hh in range(H):
            if mode == oracle.ZERO:
                ks = torch.zeros(1, d, dtype=q.dtype)
                vs = torch.zeros(1, d, dtype=q.dtype)
            elif mode == oracle.COPY_FIRST:
                ks, vs = k[b, hh, :1], v[b, hh, :1]
            else:
                ks, vs = k0[hh:hh + 1], v0[hh:hh + 1]
            K = torch.cat([ks, k[b, hh]], 0)
            V = torch.cat([vs, v[b, hh]], 0)
            for r in range(T):
                t = r + 1
                a = scale * (K[:t + 1] @ q[b, hh, r])

                def lphi2(x):
                    small = x.abs() < 0.1
                    xs = torch.where(small, x, torch.zeros_like(x))
                    xl = torch.where(small, torch.ones_like(x), x)
                    ser = sum(xs ** n / math.factorial(n + 2) for n in range(12))
                    direct = (torch.expm1(xl) - xl) / xl ** 2
                    return torch.log(torch.where(small, ser, direct))

                left = lphi2(a[:-2] - a[1:-1])
                right = lphi2(a[2:] - a[1:-1])
                b_mid = torch.logaddexp(left, right)
                b_all = torch.cat([lphi2(a[1:2] - a[0:1]), b_mid, lphi2(a[t - 1:t] - a[t:t + 1])])
                w = torch.softmax(a + b_all, 0)
                outs.append(w @ V[:t + 1])
    return torch.stack(outs).reshape(B, H, T, d)


@pytest.mark.parametrize("mode", MODES)
def test_backward_matches_autograd(mode):
    x = make_inputs(2, 2, 7, 4, "f32", seed=21 + mode)
    g = torch.randn(2, 2, 7, 4, generator=torch.Generator().manual_seed(8))
    scale = 0.9
    ref = oracle.backward(x["q"], x["k"], x["v"], g, x["k0"], x["v0"], scale=scale, mode=mode)
    leaves = {n: x[n].double().clone().requires_grad_(True) for n in ("q", "k", "v", "k0", "v0")}
    o = _torch_forward(leaves["q"], leaves["k"], leaves["v"], leaves["k0"], leaves["v0"], scale,
                       mode)
    (o * g.double()).sum().backward()
    for n in ("q", "k", "v"):
        assert np.abs(ref["d" + n] - leaves[n].grad.numpy()).max() < 1e-11, n
    if mode == oracle.GIVEN:
        for n in ("k0", "v0"):
            assert np.abs(ref["d" + n] - leaves[n].grad.numpy()).max() < 1e-11, n
    else:
        assert ref["dk0"] is None and ref["dv0"] is None


def test_backward_translation_invariants():
    # mode GIVEN: shifting every key and k0 by c leaves every logit's row
    # translated by q.c, so o and L do not move: sum dk + dk0 = 0.  Shifting
    # every value and v0 by c moves every o_t by c: sum dv + dv0 = sum dout.
    x = make_inputs(3, 2, 9, 5, "f32", seed=33)
    g = torch.randn(3, 2, 9, 5, generator=torch.Generator().manual_seed(9))
    r = oracle.backward(x["q"], x["k"], x["v"], g, x["k0"], x["v0"], scale=0.8, mode=oracle.GIVEN)
    assert np.abs(r["dk"].sum(axis=(0, 2)) + r["dk0"]).max() < 1e-12
    assert np.abs(r["dv"].sum(axis=(0, 2)) + r["dv0"] - g.double().numpy().sum(axis=(0, 2))).max() < 1e-12
    # scale = 0: every logit is 0, the weights are constant, so q and k get
    # no gradient
    for mode in MODES:
        z = oracle.backward(x["q"], x["k"], x["v"], g, x["k0"], x["v0"], scale=0.0, mode=mode)
        assert np.abs(z["dq"]).max() == 0.0 and np.abs(z["dk"]).max() == 0.0
