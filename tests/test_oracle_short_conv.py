"""Pins of the short-conv reading of eq. (13) (oracle.forward_short_conv).

eq. (13) expands b_{t,i} to first order: b_i = (a_{i-1} + a_{i+1} - 2 a_i)/6
inside the row, and the one-sided ends follow from log phi2(x) = -log 2 + x/3
+ O(x^2).  Pinned by:
  * the first row (keys 0 and 1) in closed form, worked by hand;
  * equal logits (scale 0): the same trapezoid weights as the exact method;
  * second-order agreement with the exact eq. (8) oracle: as the logit
    spread shrinks by 2, the difference shrinks by 4 (a wrong first-order
    coefficient would leave a factor 2).
"""
import math

import numpy as np
import pytest

import oracle
from continuous_softmax_attention_gb300.inputs import make_inputs


def test_first_row_closed_form():
    # t = 1, zero sink: z_0 = -log2 + a_1/3, z_1 = a_1 - log2 - a_1/3, so
    # o = v_1 e^{z_1}/(e^{z_0} + e^{z_1}) = v_1 / (1 + e^{-a_1/3})
    x = make_inputs(1, 2, 4, 8, "f32", seed=3)
    scale = 0.7
    o, lse = oracle.forward_short_conv(x["q"], x["k"], x["v"], scale=scale)
    for h in range(2):
        a1 = scale * float(np.dot(x["q"][0, h, 0].double().numpy(), x["k"][0, h, 0].double().numpy()))
        want = x["v"][0, h, 0].double().numpy() / (1.0 + math.exp(-a1 / 3.0))
        assert np.abs(o[0, h, 0] - want).max() < 1e-14
        want_lse = math.log(0.5 * math.exp(a1 / 3.0) + 0.5 * math.exp(2.0 * a1 / 3.0))
        assert abs(lse[0, h, 0] - want_lse) < 1e-14


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_equal_logits_match_exact(mode):
    x = make_inputs(1, 2, 9, 4, "f32", seed=4)
    o, lse = oracle.forward_short_conv(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.0, mode=mode)
    oe, le = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.0, mode=mode)
    assert np.abs(o - oe).max() < 1e-14 and np.abs(lse - le).max() < 1e-14


@pytest.mark.parametrize("mode", [0, 2])
def test_second_order_agreement_with_exact(mode):
    x = make_inputs(1, 2, 40, 16, "f32", seed=5)
    errs = []
    for s in (0.04, 0.02, 0.01):
        o, lse = oracle.forward_short_conv(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=s, mode=mode)
        oe, le = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=s, mode=mode)
        errs.append((np.abs(o - oe).max(), np.abs(lse - le).max()))
    for (eo1, el1), (eo2, el2) in zip(errs, errs[1:]):
        assert 3.6 < eo1 / eo2 < 4.4, errs
        assert 3.6 < el1 / el2 < 4.4, errs
