"""Ordering of the forward kernel's epilogue against the next query tile.

Each persistent CTA runs its query tiles one after another.  The two column
halves of a row keep their own accumulators O_0 and O_1, and in a tile's
epilogue every softmax thread reads both (its half's output columns of
each).  The next tile's first PV product overwrites O_0 and O_1, so the
kernel issues it only after every softmax thread has read them.  These
tests plant a delay before the reads of one column half
(csa_selftest_forward_delay) while the other half runs ahead into the next
query tile, and require the output and lse to equal an undelayed launch's
bit for bit.  A kernel without that ordering reads an accumulator the next
tile has already overwritten: a build of it failed every delay_half = 1 case
here (35,808 to 46,080 rows differ).  Its delay_half = 0 cases pass, since
the MMA thread issues each tile's half-0 product before the half-1 one, so
half 1 cannot overtake a delayed half 0; they stay as the mirror case."""
import math

import pytest
import torch

import continuous_softmax_attention_gb300 as csa
from continuous_softmax_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

# (B, H, T, d, mode): 3 to 4 query tiles per CTA on 152 SMs, both head sizes,
# the given sink (its fp32 share is added in the epilogue) and the zero sink
SHAPES = [(2, 16, 2048, 128, 0), (1, 8, 8192, 64, 2), (1, 16, 4000, 128, 2)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("half", [0, 1])
def test_delayed_epilogue_reads_give_the_same_bits(shape, half):
    B, H, T, d, mode = shape
    x = make_inputs(B, H, T, d, "bf16", seed=7)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode,
                                 scale=scale)
    o, lse = csa.selftest_forward_delay(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode,
                                        scale=scale, delay_ns=20000, delay_half=half)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    assert torch.isfinite(o.float()).all()
    bad = (o != o_ref).any(dim=-1)
    assert not bad.any(), f"{int(bad.sum())} rows differ, first at {bad.nonzero()[0].tolist()}"
    assert torch.equal(lse, lse_ref)


def test_delay_zero_is_the_plain_forward():
    B, H, T, d, mode = 1, 4, 1000, 128, 1
    x = make_inputs(B, H, T, d, "bf16", seed=8)
    g = {k: t.cuda() for k, t in x.items()}
    o_ref, lse_ref = csa.forward(g["q"], g["k"], g["v"], mode=mode)
    o, lse = csa.selftest_forward_delay(g["q"], g["k"], g["v"], mode=mode, delay_ns=0)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
