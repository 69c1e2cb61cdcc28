"""Context-parallel decode on one GPU: csa_decode_range over the ranges of a
split of the positions 0..T, each from its own cache shard, then
csa_decode_merge_ranges.

Every range's partial (fp32 o_r and lse_r) is checked against the oracle's
decode over the same positions (oracle.decode_range), and the merged result
against the oracle's whole decode row and against csa_decode.  Splits put
range edges at the kernel's chunk edges and next to the sink, and lengths
make some ranges empty for some sequences."""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import (decode, decode_merge_ranges, decode_range,
                                                decode_range_workspace_bytes)
from continuous_softmax_attention_gb300.dist import cache_shard, context_ranges
from continuous_softmax_attention_gb300.inputs import decode_workload_inputs, make_decode_inputs
from gpu_util import BF16_MAX, BF16_MEAN, LSE_TOL, np64

pytestmark = pytest.mark.gpu

PART_TOL = 1e-4  # fp32 partials from bf16 inputs: fp32 arithmetic throughout


def chunk(d):
    """Positions per chunk of the decode kernel (staged keys minus the two halo keys)."""
    return (112 if d == 256 else 16384 // d) - 2


def run_ranges(x, T, ranges, scale, mode):
    dev = {k: t.cuda() for k, t in x.items() if k != "seqlens"}
    sl = torch.as_tensor(x["seqlens"], dtype=torch.int32).cuda()
    parts = []
    for lo, hi in ranges:
        ks, vs = cache_shard(dev["k"], dev["v"], lo, hi)
        parts.append(decode_range(dev["q"], ks, vs, T, lo, hi, dev["k0"], dev["v0"], seqlens=sl,
                                  mode=mode, scale=scale))
    o_parts = torch.stack([o for o, _ in parts])
    l_parts = torch.stack([l for _, l in parts])
    o, lse = decode_merge_ranges(o_parts, l_parts)
    full = decode(dev["q"], dev["k"], dev["v"], dev["k0"], dev["v0"], seqlens=sl, mode=mode,
                  scale=scale)
    torch.cuda.synchronize()
    return parts, (o, lse), full


def splits(T, d):
    C = chunk(d)
    out = [context_ranges(T, R) for R in (2, 3, 5)]
    out.append([(0, 2), (2, C), (C, T + 1)])  # the sink and key 1 alone
    out.append([(0, C - 1), (C - 1, C + 1), (C + 1, 2 * C + 3), (2 * C + 3, T + 1)])
    return out


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_ranges_merge_to_the_decode_step(d, mode):
    C = chunk(d)
    T = 2 * C + 40
    x = make_decode_inputs(4, 2, T, d, 31 + d + mode, 1)
    x["seqlens"] = torch.tensor([T, 1, C + 1, 2 * C - 1], dtype=torch.int32)
    scale = d ** -0.5
    ro, rl = oracle.decode_range(x["q"], x["k"], x["v"], x["seqlens"], 0, T + 1, x["k0"],
                                 x["v0"], scale=scale, mode=mode)
    for ranges in splits(T, d):
        parts, (o, lse), (fo, fl) = run_ranges(x, T, ranges, scale, mode)
        for (lo, hi), (po, pl) in zip(ranges, parts):
            eo, el = oracle.decode_range(x["q"], x["k"], x["v"], x["seqlens"], lo, hi, x["k0"],
                                         x["v0"], scale=scale, mode=mode)
            po, pl = np64(po), np64(pl)
            empty = np.isneginf(el)
            assert (np.isneginf(pl) == empty).all(), (lo, hi)
            assert (po[empty] == 0).all()
            assert np.abs(po[~empty] - eo[~empty]).max(initial=0) <= PART_TOL, (lo, hi)
            assert np.abs(pl[~empty] - el[~empty]).max(initial=0) <= PART_TOL, (lo, hi)
        o, lse = np64(o), np64(lse)
        err = np.abs(o - ro)
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, ranges
        assert np.abs(lse - rl).max() <= LSE_TOL, ranges
        # the same result as the single-device step, up to the bf16 rounding of o
        assert np.abs(o - np64(fo)).max() <= 2 ** -7 * max(np.abs(ro).max(), 1.0), ranges
        assert np.abs(lse - np64(fl)).max() <= 1e-5, ranges


def test_timed_decode_workload_split_over_four_ranges():
    """The 16 x 32 x 8192 x 128 decode workload split into four ranges: the
    merged step equals csa_decode's (sampled against the oracle there)."""
    x = decode_workload_inputs("decode")
    T, d = x["k"].shape[2], x["k"].shape[3]
    ranges = context_ranges(T, 4)
    for lo, hi in ranges:
        assert decode_range_workspace_bytes(16, 32, lo, hi, d) > 0
    parts, (o, lse), (fo, fl) = run_ranges(x, T, ranges, d ** -0.5, 0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert (o.float() - fo.float()).abs().max().item() <= 2 ** -7 * max(fo.float().abs().max().item(), 1.0)
    assert (lse - fl).abs().max().item() <= 1e-5
