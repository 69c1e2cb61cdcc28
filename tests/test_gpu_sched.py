"""Scheduling of the persistent tensor-core forward kernel.

The kernel runs one CTA per SM and takes query tiles from a counter; each
launch uses one of 64 counter slots, reused in turn, with reuse ordered by an
event per slot.  A query tile is computed by one CTA from start to end in a
fixed order, so whichever CTA takes it, the result is the same bits.  These
tests run launches on several streams at once, more launches than there are
slots, and grids smaller than the SM count, and compare every result with a
launch made alone."""
import math

import pytest
import torch

import continuous_softmax_attention_gb300 as csa
from continuous_softmax_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

# (B, H, T, d, mode): several items per SM, fewer items than SMs, one item,
# a ragged tail, both head sizes, all three sink modes
SHAPES = [(1, 8, 2048, 128, 0), (2, 3, 300, 64, 1), (1, 1, 100, 128, 2), (1, 4, 1000, 64, 2)]


def _inputs(i, shape):
    B, H, T, d, mode = shape
    x = make_inputs(B, H, T, d, "bf16", seed=100 + i)
    return {k: t.cuda() for k, t in x.items()}, mode, 1.0 / math.sqrt(d)


def _forward(g, mode, scale, form):
    if form == "symmetric":
        return csa.forward_symmetric(g["q"], g["k"], g["v"], scale=scale)
    return csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale,
                       short_conv=form == "short_conv")


@pytest.mark.parametrize("form", ["exact", "short_conv", "symmetric"])
def test_concurrent_streams_and_slot_reuse_match_single_launches(form):
    cases = [_inputs(i, s) for i, s in enumerate(SHAPES)]
    ref = []
    for g, mode, scale in cases:
        o, lse = _forward(g, mode, scale, form)
        torch.cuda.synchronize()
        ref.append((o.clone(), lse.clone()))
    streams = [torch.cuda.Stream() for _ in cases]
    outs = []
    # 4 streams x 20 rounds = 80 launches: every slot is reused, some while
    # launches of other streams are in flight
    for _ in range(20):
        for (g, mode, scale), st in zip(cases, streams):
            with torch.cuda.stream(st):
                outs.append(_forward(g, mode, scale, form))
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    for n, (o, lse) in enumerate(outs):
        ro, rl = ref[n % len(cases)]
        assert torch.equal(o, ro), n
        assert torch.equal(lse, rl), n


def test_many_back_to_back_launches_one_stream():
    """More launches than slots on one stream, each writing its own output."""
    g, mode, scale = _inputs(0, SHAPES[0])
    ro, rl = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale)
    outs = [csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale)
            for _ in range(150)]
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    for o, lse in outs:
        assert torch.equal(o, ro) and torch.equal(lse, rl)


@pytest.mark.parametrize("H, T", [(19, 1024), (17, 1152), (1, 19456), (3, 6400)])
def test_item_counts_around_the_sm_count(H, T):
    """Query tiles: 19 x 8 = 152 (one per CTA on a 152-SM part), 17 x 9 =
    153 (one CTA takes a second), 152 in one head, 150 over three heads.
    Every head of one launch is bit-identical to that head launched alone,
    where each CTA holds at most one query tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x = make_inputs(1, H, T, 128, "bf16", seed=7 + H)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 128 ** -0.5
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=2, scale=scale)
    for h in range(H):
        sl = lambda t: t[:, h:h + 1].contiguous()
        oh, lh = csa.forward(sl(g["q"]), sl(g["k"]), sl(g["v"]), g["k0"][h:h + 1].contiguous(),
                             g["v0"][h:h + 1].contiguous(), mode=2, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o[:, h:h + 1], oh), (h, sms)
        assert torch.equal(lse[:, h:h + 1], lh), (h, sms)
    assert csa.device_status() == 0
