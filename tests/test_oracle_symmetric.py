"""Pins of the symmetric-interval oracle (oracle.forward_symmetric): eq. (2)
over [1/2, t + 1/2] with eq. (3) inside [1, t] and constant end half-cells.

  * composite Gauss-Legendre quadrature of the two integrals themselves
    (oracle.quadrature.forward_symmetric, no phi function);
  * equal logits: every token owns a unit cell, so o_t is the plain mean of
    v_1..v_t and lse_t = log t;
  * t = 1: the single half-open cell [1/2, 3/2] holds v_1, so o_1 = v_1.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import quadrature
from continuous_softmax_attention_gb300.inputs import make_inputs


@pytest.mark.parametrize("scale", [0.3, 1.5, 6.0])
def test_symmetric_matches_quadrature(scale):
    x = make_inputs(2, 2, 11, 5, "f32", seed=30)
    o, lse = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=scale)
    qo, ql = quadrature.forward_symmetric(x["q"].numpy(), x["k"].numpy(), x["v"].numpy(), scale=scale)
    assert np.abs(o - qo).max() < 1e-12 and np.abs(lse - ql).max() < 1e-12


def test_symmetric_equal_logits_is_the_mean():
    x = make_inputs(1, 3, 13, 4, "f32", seed=31)
    o, lse = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=0.0)
    v = x["v"].double().numpy()
    for r in range(13):
        assert np.abs(o[0, :, r] - v[0, :, :r + 1].mean(axis=1)).max() < 1e-14
        assert np.abs(lse[0, :, r] - math.log(r + 1)).max() < 1e-14


def test_symmetric_first_row():
    x = make_inputs(2, 2, 5, 7, "f32", seed=32)
    o, lse = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=0.9)
    assert np.abs(o[:, :, 0] - x["v"][:, :, 0].double().numpy()).max() < 1e-15
    a = 0.9 * (x["q"][:, :, 0].double() * x["k"][:, :, 0].double()).sum(-1).numpy()
    assert np.abs(lse[:, :, 0] - a).max() < 1e-13


def test_symmetric_rows_match_full():
    x = make_inputs(2, 2, 30, 8, "f32", seed=33)
    o, lse = oracle.forward_symmetric(x["q"], x["k"], x["v"], scale=0.6)
    picks = [(1, 0, 0), (0, 1, 29), (1, 1, 17)]
    ro, rl = oracle.forward_symmetric_rows(x["q"], x["k"], x["v"], oracle.flat_rows(2, 2, 30, picks),
                                           scale=0.6)
    for n, (b, h, r) in enumerate(picks):
        assert np.array_equal(ro[n], o[b, h, r]) and rl[n] == lse[b, h, r]
