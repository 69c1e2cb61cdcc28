"""Decode step (csa_decode) against the CPU oracle.

The decode output of sequence b is row n_b - 1 of eq. (8) over the first n_b
tokens; the oracle computes exactly that row, from the same bf16 values, on
a [1, 1, n_b, d] slice whose last query row is the decode query.  Lengths are
picked around the kernel's chunk edges (C = 16384 / d - 2 positions, position 0
being the sink), so that the halo keys across chunks and the one-sided end
terms of eq. (10) are all exercised."""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import CsaError, decode, decode_workspace_bytes, device_status
from continuous_softmax_attention_gb300 import forward
from continuous_softmax_attention_gb300.inputs import (DECODE_WORKLOADS, decode_workload_inputs,
                                                       make_decode_inputs)
from gpu_util import BF16_MAX, BF16_MEAN, LSE_TOL, np64

pytestmark = pytest.mark.gpu


def chunk(d):
    """Positions per chunk of the decode kernel (staged keys minus the two halo keys)."""
    return (112 if d == 256 else 16384 // d) - 2


def oracle_decode(x, seqlens, scale, mode, pairs):
    """Row n_b - 1 of eq. (8) for each (b, h) in pairs."""
    d = x["k"].shape[-1]
    os_, ls = [], []
    for b, h in pairs:
        n = int(seqlens[b])
        qf = torch.zeros(1, 1, n, d, dtype=torch.float32)
        qf[0, 0, n - 1] = x["q"][b, h].float()
        o, lse = oracle.forward_rows(qf, x["k"][b:b + 1, h:h + 1, :n], x["v"][b:b + 1, h:h + 1, :n],
                                     [n - 1], k0=x["k0"][h:h + 1], v0=x["v0"][h:h + 1],
                                     scale=scale, mode=mode)
        os_.append(o[0])
        ls.append(lse[0])
    return np.stack(os_), np.asarray(ls)


def run_decode(x, seqlens, scale, mode, **kw):
    dev = {k: t.cuda() for k, t in x.items() if k != "seqlens"}
    sl = torch.as_tensor(seqlens, dtype=torch.int32).cuda()
    o, lse = decode(dev["q"], dev["k"], dev["v"], dev["k0"], dev["v0"], seqlens=sl, mode=mode,
                    scale=scale, **kw)
    torch.cuda.synchronize()
    return o, lse


def check(o, lse, ro, rl, what):
    o, lse = np64(o), np64(lse)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    err, lerr = np.abs(o - ro), np.abs(lse - rl)
    assert err.max() <= BF16_MAX, f"{what}: max |o err| {err.max():.3g}"
    assert err.mean() <= BF16_MEAN, f"{what}: mean |o err| {err.mean():.3g}"
    assert lerr.max() <= LSE_TOL, f"{what}: max |lse err| {lerr.max():.3g}"


def edge_lengths(d, T):
    C = chunk(d)
    return [n for n in (1, 2, 3, C - 2, C - 1, C, C + 1, 2 * C - 1, 2 * C, T) if 1 <= n <= T]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_decode_chunk_edges(d, mode):
    T = 3 * chunk(d) + 5
    lens = edge_lengths(d, T)
    x = make_decode_inputs(len(lens), 2, T, d, seed=20 + d + mode)
    pairs = [(b, h) for b in range(len(lens)) for h in range(2)]
    scale = 1.0 / d ** 0.5
    o, lse = run_decode(x, lens, scale, mode)
    ro, rl = oracle_decode(x, lens, scale, mode, pairs)
    check(o.reshape(-1, d), lse.reshape(-1), ro, rl, f"d={d} mode={mode}")


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0, -0.5])
def test_decode_logit_ranges(scale):
    # scale 4 at d = 64 gives logit gaps of order +-100 between neighbours
    d, T = 64, 700
    C = chunk(d)
    lens = [1, C - 1, C, C + 1, 2 * C + 1, T]
    x = make_decode_inputs(len(lens), 3, T, d, seed=31)
    pairs = [(b, h) for b in range(len(lens)) for h in range(3)]
    o, lse = run_decode(x, lens, scale, 0)
    ro, rl = oracle_decode(x, lens, scale, 0, pairs)
    check(o.reshape(-1, d), lse.reshape(-1), ro, rl, f"scale={scale}")


def test_decode_small_workload_all_modes():
    w = DECODE_WORKLOADS["decode_small"]
    x = decode_workload_inputs("decode_small")
    lens = x["seqlens"].tolist()
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    for mode in (0, 1, 2):
        o, lse = run_decode(x, lens, None, mode)
        ro, rl = oracle_decode(x, lens, 1.0 / w.d ** 0.5, mode, pairs)
        check(o.reshape(-1, w.d), lse.reshape(-1), ro, rl, f"mode={mode}")


def test_decode_full_workload_sampled():
    """The timed decode workload, checked on sampled (b, h) pairs."""
    w = DECODE_WORKLOADS["decode"]
    x = decode_workload_inputs("decode")
    lens = x["seqlens"].tolist()
    o, lse = run_decode(x, lens, None, w.mode)
    rng = np.random.default_rng(7)
    pairs = [(int(b), int(h)) for b, h in zip(rng.integers(0, w.B, 12), rng.integers(0, w.H, 12))]
    pairs += [(0, 0), (w.B - 1, w.H - 1)]
    ro, rl = oracle_decode(x, lens, 1.0 / w.d ** 0.5, w.mode, pairs)
    idx_b = [b for b, _ in pairs]
    idx_h = [h for _, h in pairs]
    check(o[idx_b, idx_h], lse[idx_b, idx_h], ro, rl, "decode workload")


def test_decode_matches_forward_last_row():
    """Same row by the tensor-core forward kernel (which rounds the weights to
    bf16 for the tensor core): agreement within the bf16 bar."""
    B, H, T, d = 2, 4, 300, 128
    x = make_decode_inputs(B, H, T, d, seed=41)
    qfull = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    qfull[:, :, T - 1] = x["q"]
    for mode in (0, 1, 2):
        fo, fl = forward(qfull.cuda(), x["k"].cuda(), x["v"].cuda(), x["k0"].cuda(),
                         x["v0"].cuda(), mode=mode)
        o, lse = run_decode(x, [T] * B, 1.0 / d ** 0.5, mode)
        err = (o.float() - fo[:, :, T - 1].float()).abs()
        assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN
        assert (lse - fl[:, :, T - 1]).abs().max().item() <= LSE_TOL


def test_decode_full_length_without_seqlens():
    B, H, T, d = 2, 2, 400, 128
    x = make_decode_inputs(B, H, T, d, seed=43)
    dev = {k: t.cuda() for k, t in x.items() if k != "seqlens"}
    o, lse = decode(dev["q"], dev["k"], dev["v"])
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    ro, rl = oracle_decode(x, [T] * B, 1.0 / d ** 0.5, 0, pairs)
    check(o.reshape(-1, d), lse.reshape(-1), ro, rl, "seqlens=None")


def test_decode_deterministic_and_ignores_stale_workspace():
    B, H, T, d = 3, 4, 1000, 128
    x = make_decode_inputs(B, H, T, d, seed=44, len_lo=100)
    ws = torch.full((decode_workspace_bytes(B, H, T, d) // 4,), float("nan"), device="cuda")
    o1, l1 = run_decode(x, x["seqlens"].tolist(), None, 0, workspace=ws)
    o2, l2 = run_decode(x, x["seqlens"].tolist(), None, 0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_length_out_of_range_sets_status():
    B, H, T, d = 3, 2, 200, 64
    x = make_decode_inputs(B, H, T, d, seed=45)
    assert device_status() == 0
    o, lse = run_decode(x, [0, 150, T + 1], None, 0)
    assert device_status() == -1  # CSA_ERR_INVALID_ARG, then cleared
    assert device_status() == 0
    assert torch.isnan(o[0].float()).all() and torch.isnan(o[2].float()).all()
    assert torch.isnan(lse[0]).all() and torch.isnan(lse[2]).all()
    ro, rl = oracle_decode(x, [0, 150, 0], 1.0 / d ** 0.5, 0, [(1, 0), (1, 1)])
    check(o[1], lse[1], ro, rl, "valid sequence next to invalid ones")


def test_decode_argument_errors():
    x = make_decode_inputs(1, 1, 64, 128, seed=46)
    dev = {k: t.cuda() for k, t in x.items() if k != "seqlens"}
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(CsaError) as e:
        decode(dev["q"], dev["k"], dev["v"], workspace=small)
    assert e.value.code == -1
    with pytest.raises(ValueError):
        decode(dev["q"], dev["k"], dev["v"], mode=2)
    o, lse = decode(dev["q"][:0], dev["k"][:0], dev["v"][:0])  # empty batch
    assert o.shape == (0, 1, 128)


def test_decode_very_long_cache():
    """One sequence of 131072 cached keys (1041 chunks) next to a short one."""
    B, H, T, d = 2, 2, 131072, 128
    x = make_decode_inputs(B, H, T, d, seed=510, len_lo=T)
    lens = [T, 1000]
    o, lse = run_decode(x, lens, None, 2)
    ro, rl = oracle_decode(x, lens, 1.0 / d ** 0.5, 2, [(0, 0), (0, 1), (1, 0), (1, 1)])
    check(o.reshape(-1, d), lse.reshape(-1), ro, rl, "T=131072")
