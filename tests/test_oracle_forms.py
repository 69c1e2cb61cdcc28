"""Pins of the oracle's attention forms against the definitions and the
mathematics of "Continuous Softmax Attention" (Jianlin Su) and of standard
causal attention ("Attention, from the softmax up", section "In code").

Every check compares the closed-form oracle with something independent of
it: quadrature of eq. (2), 50-digit evaluation of the segment integrals,
torch's scaled_dot_product_attention, exact closed forms of special cases,
invariances, and the Taylor expansion (13)."""
import math

import mpmath
import numpy as np
import pytest
import torch

import oracle
from oracle import quadrature
from continuous_softmax_attention_gb300.inputs import make_inputs

ZERO, COPY_FIRST, GIVEN = oracle.ZERO, oracle.COPY_FIRST, oracle.GIVEN
MODES = [ZERO, COPY_FIRST, GIVEN]


def _inp(B, H, T, d, seed, dtype="f32"):
    x = make_inputs(B, H, T, d, dtype, seed)
    return {kk: vv.float().numpy() for kk, vv in x.items()}


@pytest.mark.parametrize("mode", MODES)
def test_quadrature_tiny_workload(mode):
    """eq. (8) == eq. (2) by quadrature on the tiny workload (T=64, d=16, scale 1/4)."""
    x = _inp(1, 1, 64, 16, 0)
    o8, l8 = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.25, mode=mode)
    oq, lq = quadrature.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.25, mode=mode)
    assert np.max(np.abs(o8 - oq)) < 1e-10
    assert np.max(np.abs(l8 - lq)) < 1e-10


@pytest.mark.parametrize("scale", [0.5, 2.0, 6.0])
@pytest.mark.parametrize("mode", MODES)
def test_quadrature_large_gaps(scale, mode):
    """Large logit gaps exercise the log-domain branches of phi1/phi2."""
    x = _inp(1, 2, 12, 8, 7)
    o8, l8 = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    oq, lq = quadrature.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    assert np.max(np.abs(o8 - oq)) < 1e-9
    assert np.max(np.abs(l8 - lq)) < 1e-9


def test_segment_integrals_high_precision():
    """eq. (4)/(5) for each unit interval, integrated in 50-digit arithmetic
    (mpmath.quad over the interpolated k_s, v_s), with logit gaps up to ~100."""
    mpmath.mp.dps = 50
    x = _inp(1, 1, 5, 3, 11)
    scale = 20.0
    o8, l8 = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=GIVEN)
    q, k, v = x["q"][0, 0], x["k"][0, 0], x["v"][0, 0]
    K = np.vstack([x["k0"][0:1], k]).astype(np.float64)
    V = np.vstack([x["v0"][0:1], v]).astype(np.float64)
    for r in range(5):
        t = r + 1
        qt = [mpmath.mpf(float(c)) for c in q[r]]
        a = [scale * mpmath.fsum(qt[c] * mpmath.mpf(K[i][c]) for c in range(3)) for i in range(t + 1)]
        num = [mpmath.mpf(0)] * 3
        den = mpmath.mpf(0)
        for i in range(1, t + 1):
            f = lambda s, i=i: mpmath.exp((1 - s) * a[i - 1] + s * a[i])
            den += mpmath.quad(f, [0, 1])
            for c in range(3):
                num[c] += mpmath.quad(lambda s, i=i, c=c: f(s) * ((1 - s) * V[i - 1][c] + s * V[i][c]), [0, 1])
        for c in range(3):
            assert o8[0, 0, r, c] == pytest.approx(float(num[c] / den), rel=1e-12, abs=1e-13)
        assert l8[0, 0, r] == pytest.approx(float(mpmath.log(den)), rel=1e-13, abs=1e-13)


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0])
@pytest.mark.parametrize("mode", MODES)
def test_eq8_equals_eq11(scale, mode):
    """The re-indexing (9) turns the segment sum (8) into the softmax form (11)."""
    x = _inp(2, 2, 40, 8, 3)
    o8, l8 = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    o11, l11 = oracle.forward_eq11(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)
    assert np.max(np.abs(o8 - o11)) < 1e-12
    assert np.max(np.abs(l8 - l11)) < 1e-12


@pytest.mark.parametrize("mode", MODES)
def test_equal_logits_trapezoid(mode):
    """scale = 0 makes every logit equal: interior weights 1, end weights 1/2
    (phi2(0) = 1/2), i.e. the trapezoid rule:
    o_t = (v0/2 + v_1 + ... + v_{t-1} + v_t/2) / t and lse_t = log t."""
    x = _inp(1, 2, 17, 5, 5)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.0, mode=mode)
    for h in range(2):
        v = x["v"][0, h].astype(np.float64)
        v0 = {ZERO: np.zeros(5), COPY_FIRST: v[0], GIVEN: x["v0"][h].astype(np.float64)}[mode]
        V = np.vstack([v0[None], v])
        for r in range(17):
            t = r + 1
            expect = (0.5 * V[0] + V[1:t].sum(axis=0) + 0.5 * V[t]) / t
            assert np.max(np.abs(o[0, h, r] - expect)) < 1e-13
            assert lse[0, h, r] == pytest.approx(math.log(t), abs=1e-13)


def test_copy_first_sink_bias_is_log_half():
    """k_0 = k_1 gives a_{t,0} = a_{t,1}, so e^{b_{t,0}} = phi2(0) = 1/2."""
    x = _inp(1, 1, 30, 6, 9)
    for r in (0, 1, 7, 29):
        a, b = oracle.row_bias(x["q"], x["k"], 0, 0, r, scale=0.7, mode=COPY_FIRST)
        assert a[0] == a[1]
        assert b[0] == pytest.approx(math.log(0.5), abs=1e-15)


def test_key_translation_invariance():
    """Adding u to every key (and to k_0) adds scale*q_t.u to every logit of
    row t: o is unchanged and lse_t moves by scale*q_t.u."""
    x = _inp(1, 2, 25, 6, 13)
    u = np.random.default_rng(0).standard_normal(6).astype(np.float32) * 0.5
    scale = 0.8
    o1, l1 = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=GIVEN)
    # The oracle reads float32, so k + u is rounded to float32 (relative 6e-8);
    # the tolerance below covers that rounding and nothing else.
    k2 = (x["k"] + u).astype(np.float32)
    k02 = (x["k0"] + u).astype(np.float32)
    o2, l2 = oracle.forward(x["q"], k2, x["v"], k02, x["v0"], scale=scale, mode=GIVEN)
    shift = scale * np.einsum("bhtd,d->bht", x["q"].astype(np.float64), u.astype(np.float64))
    assert np.max(np.abs(o1 - o2)) < 1e-5
    assert np.max(np.abs((l2 - l1) - shift)) < 1e-5


def test_causality():
    """Changing keys/values after position t leaves rows <= t unchanged."""
    x = _inp(1, 1, 40, 8, 17)
    o1, l1 = oracle.forward(x["q"], x["k"], x["v"], scale=0.9)
    k2, v2 = x["k"].copy(), x["v"].copy()
    cut = 23
    k2[0, 0, cut + 1:] += 3.0
    v2[0, 0, cut + 1:] -= 5.0
    o2, l2 = oracle.forward(x["q"], k2, v2, scale=0.9)
    assert np.array_equal(o1[0, 0, :cut + 1], o2[0, 0, :cut + 1])
    assert np.array_equal(l1[0, 0, :cut + 1], l2[0, 0, :cut + 1])
    assert not np.array_equal(o1[0, 0, cut + 1:], o2[0, 0, cut + 1:])


@pytest.mark.parametrize("mode", [COPY_FIRST, GIVEN])
def test_constant_values(mode):
    """If every v_i (the sink's v_0 included) equals c, eq. (11) gives o_t = c."""
    x = _inp(1, 2, 33, 4, 19)
    c = np.array([0.25, -1.5, 3.0, 0.0], dtype=np.float32)
    v = np.broadcast_to(c, x["v"].shape).copy()
    v0 = np.broadcast_to(c, x["v0"].shape).copy()
    o, _ = oracle.forward(x["q"], x["k"], v, x["k0"], v0, scale=1.3, mode=mode)
    assert np.max(np.abs(o - c)) < 1e-13


def test_zero_sink_shrinks_constant_values():
    """With k_0 = v_0 = 0 the sink pulls o toward 0: o_t = c * (1 - w_0/W)."""
    x = _inp(1, 1, 10, 4, 23)
    c = np.float32(2.0)
    v = np.full(x["v"].shape, c, dtype=np.float32)
    o, _ = oracle.forward(x["q"], x["k"], v, scale=0.5, mode=ZERO)
    assert np.all(o < c) and np.all(o > 0)


@pytest.mark.parametrize("scale", [0.3, 3.0, 30.0])
def test_weight_bound(scale):
    """e^{a_i + b_i} <= max(e^{a_{i-1}}, e^{a_i}, e^{a_{i+1}}): each phi2 term
    is the integral of e^{(convex combination)} (1-s) <= max/2."""
    x = _inp(1, 1, 64, 8, 29)
    for r in (0, 1, 5, 31, 63):
        a, b = oracle.row_bias(x["q"], x["k"], 0, 0, r, scale=scale)
        t = r + 1
        for i in range(t + 1):
            nb = [a[j] for j in (i - 1, i, i + 1) if 0 <= j <= t]
            assert a[i] + b[i] <= max(nb) + 1e-12


def test_taylor_expansion_13():
    """eq. (13): b_i = (a_{i-1} + a_{i+1} - 2 a_i)/6 + ..., and the next term
    is (x^2 - x y + y^2)/36 with x = a_{i-1}-a_i, y = a_{i+1}-a_i; at the ends
    b_0 = log(1/2) + x/3 + x^2/36 with x = a_1 - a_0."""
    x = _inp(1, 1, 20, 8, 31)
    r = 19
    for eps in (1e-2, 1e-3):
        a, b = oracle.row_bias(x["q"], x["k"], 0, 0, r, scale=eps, mode=GIVEN, k0=x["k0"])
        t = r + 1
        worst1 = worst2 = 0.0
        for i in range(1, t):
            xx, yy = a[i - 1] - a[i], a[i + 1] - a[i]
            first = (a[i - 1] + a[i + 1] - 2 * a[i]) / 6.0
            second = (xx * xx - xx * yy + yy * yy) / 36.0
            worst1 = max(worst1, abs(b[i] - first))
            worst2 = max(worst2, abs(b[i] - first - second))
        scale_a = max(abs(a[i] - a[i - 1]) for i in range(1, t + 1))
        assert worst1 < 0.1 * scale_a ** 2  # first order captures all of O(eps)
        assert worst2 < 0.05 * scale_a ** 3  # second order captures all of O(eps^2)
        x0 = a[1] - a[0]
        assert abs(b[0] - (math.log(0.5) + x0 / 3 + x0 * x0 / 36)) < 0.05 * abs(x0) ** 3 + 1e-15


@pytest.mark.parametrize("scale", [None, 1.0])
def test_std_oracle_against_sdpa(scale):
    """eq. (12) matches torch's scaled_dot_product_attention (is_causal) on the
    (2, 4, 128, 64) shape of the page's check, in float64."""
    x = _inp(2, 4, 128, 64, 37)
    o, lse = oracle.std_forward(x["q"], x["k"], x["v"], scale=scale)
    q, k, v = (torch.from_numpy(x[n]).double() for n in ("q", "k", "v"))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=scale)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12
    s = (1.0 / 8.0) if scale is None else scale
    logits = (q @ k.transpose(-1, -2)) * s
    mask = torch.ones(128, 128, dtype=torch.bool).triu(1)
    ref_lse = torch.logsumexp(logits.masked_fill(mask, float("-inf")), dim=-1)
    assert np.max(np.abs(lse - ref_lse.numpy())) < 1e-12


def test_rows_entry_matches_full():
    x = _inp(2, 3, 50, 8, 41)
    o, l = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.6, mode=GIVEN)
    picks = [(0, 0, 0), (1, 2, 49), (0, 1, 17), (1, 0, 33)]
    rows = oracle.flat_rows(2, 3, 50, picks)
    orr, lr = oracle.forward_rows(x["q"], x["k"], x["v"], rows, x["k0"], x["v0"], scale=0.6, mode=GIVEN)
    for n, (b, h, r) in enumerate(picks):
        assert np.array_equal(orr[n], o[b, h, r])
        assert lr[n] == l[b, h, r]
    os_, ls_ = oracle.std_forward(x["q"], x["k"], x["v"], scale=0.6)
    orr, lr = oracle.forward_rows(x["q"], x["k"], x["v"], rows, scale=0.6, std=True)
    for n, (b, h, r) in enumerate(picks):
        assert np.array_equal(orr[n], os_[b, h, r])


def test_single_token_and_empty():
    """T = 1: token 1 sees k_0 and k_1 only; T = 0 is an empty problem."""
    x = _inp(1, 1, 1, 4, 43)
    o, l = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=1.0, mode=GIVEN)
    oq, lq = quadrature.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=1.0, mode=GIVEN)
    assert np.max(np.abs(o - oq)) < 1e-12 and np.max(np.abs(l - lq)) < 1e-12
    e = np.zeros((1, 1, 0, 4), dtype=np.float32)
    o, l = oracle.forward(e, e, e, scale=1.0)
    assert o.shape == (1, 1, 0, 4)


def test_bad_arguments_rejected():
    x = _inp(1, 1, 4, 4, 47)
    with pytest.raises(ValueError):
        oracle.forward(x["q"], x["k"], x["v"], None, None, scale=1.0, mode=GIVEN)
    with pytest.raises(ValueError):
        oracle.forward(x["q"], x["k"][:, :, :3], x["v"], scale=1.0)
