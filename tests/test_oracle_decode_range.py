"""Pins of oracle.decode_range, the decode step over a range of positions.

The range partial is eq. (11) of row t = n_b summed over some positions only
(via row_bias, the eq. (10) corrections).  It is pinned against the oracle's
decode of the whole row through a different closed form (eq. (8), the
segment sums of forward_rows): the range covering every position must give
that row, and the ranges of any partition, merged with weights e^{lse_r},
must give it too.  A planted mistake in a range's bounds, in the sink's
value or in a neighbour used for b breaks one of these."""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300.inputs import make_decode_inputs


def whole_rows(x, scale, mode):
    """Row n_b - 1 of eq. (8) (forward_rows) for every (b, h)."""
    B, H, T, d = x["k"].shape
    o = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    for b in range(B):
        n = int(x["seqlens"][b])
        for h in range(H):
            qf = torch.zeros(1, 1, n, d)
            qf[0, 0, n - 1] = x["q"][b, h].float()
            ro, rl = oracle.forward_rows(qf, x["k"][b:b + 1, h:h + 1, :n],
                                         x["v"][b:b + 1, h:h + 1, :n], [n - 1],
                                         k0=x["k0"][h:h + 1], v0=x["v0"][h:h + 1], scale=scale,
                                         mode=mode)
            o[b, h], lse[b, h] = ro[0], rl[0]
    return o, lse


def merge(parts):
    lses = np.stack([l for _, l in parts])
    L = lses.max(axis=0)
    w = np.exp(lses - L)
    o = sum(w[i][..., None] * parts[i][0] for i in range(len(parts))) / w.sum(axis=0)[..., None]
    return o, L + np.log(w.sum(axis=0))


def inputs(seed, mode):
    x = make_decode_inputs(2, 2, 200, 32, seed, 1)
    x["seqlens"] = np.array([200, 37])
    return x


@pytest.mark.parametrize("mode", [oracle.ZERO, oracle.COPY_FIRST, oracle.GIVEN])
def test_whole_range_is_the_decode_row(mode):
    x = inputs(11, mode)
    scale = 32 ** -0.5
    ro, rl = whole_rows(x, scale, mode)
    o, lse = oracle.decode_range(x["q"], x["k"], x["v"], x["seqlens"], 0, 201, x["k0"], x["v0"],
                                 scale=scale, mode=mode)
    assert np.abs(o - ro).max() < 1e-10
    assert np.abs(lse - rl).max() < 1e-10


@pytest.mark.parametrize("mode", [oracle.ZERO, oracle.COPY_FIRST, oracle.GIVEN])
@pytest.mark.parametrize("cuts", [[0, 1, 201], [0, 2, 38, 39, 201], [0, 50, 100, 150, 201],
                                  [0, 37, 38, 201]])
def test_partitions_merge_to_the_row(mode, cuts):
    """The sink alone, a range ending at a sequence's last position, ranges
    past the shorter sequence's end (empty there), single positions."""
    x = inputs(12, mode)
    scale = 1.0
    ro, rl = whole_rows(x, scale, mode)
    parts = [oracle.decode_range(x["q"], x["k"], x["v"], x["seqlens"], a, b, x["k0"], x["v0"],
                                 scale=scale, mode=mode) for a, b in zip(cuts, cuts[1:])]
    o, lse = merge(parts)
    assert np.abs(o - ro).max() < 1e-9
    assert np.abs(lse - rl).max() < 1e-9


def test_empty_range():
    x = inputs(13, oracle.ZERO)
    o, lse = oracle.decode_range(x["q"], x["k"], x["v"], x["seqlens"], 100, 150, scale=0.2)
    assert np.isneginf(lse[1]).all() and (o[1] == 0).all()  # sequence 1 has 37 tokens
    assert np.isfinite(lse[0]).all()
