"""Backward pass (csa_backward, csa_backward_f32) against the CPU oracle.

The GPU forward pass supplies out and lse (as a training step would); the
oracle recomputes everything in double from the same input values and
differentiates eq. (10)/(11) by the plain chain rule, so the comparison
covers the GPU's flux form of the gradient too.

Bars (derived from the arithmetic; the pages state none for gradients):
  fp32 inputs: normwise relative error <= 1e-5 and every element within
      1e-4 * max|ref| (fp32 rounding, amplified at most ~100x by the
      cancellations in dP - D and in the interval closed forms, summed over
      at most a few hundred keys);
  bf16 inputs: normwise relative error <= 1e-2 and every element within
      2e-2 * max|ref| (the outputs are rounded to bf16, 2^-9 relative, and
      D = dout . out uses the forward's bf16-rounded out).
"""
import numpy as np
import pytest
import torch

import oracle
from continuous_softmax_attention_gb300 import (CsaError, backward, backward_workspace_bytes,
                                                forward)
from continuous_softmax_attention_gb300.inputs import make_inputs, workload_inputs
from gpu_util import np64

pytestmark = pytest.mark.gpu

BARS = {"f32": (1e-5, 1e-4), "bf16": (1e-2, 2e-2)}


def run(x, g, scale, mode):
    dev = {k: t.cuda() for k, t in x.items()}
    gd = g.to(dev["q"].dtype).cuda()
    o, lse = forward(dev["q"], dev["k"], dev["v"], dev["k0"], dev["v0"], mode=mode, scale=scale)
    out = backward(dev["q"], dev["k"], dev["v"], o, lse, gd, dev["k0"], dev["v0"], mode=mode,
                   scale=scale)
    torch.cuda.synchronize()
    return out, gd.cpu()


def check(got, ref, dtype, what):
    norm_bar, max_bar = BARS[dtype]
    g = np64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite"
    err = np.abs(g - ref)
    scale = max(np.abs(ref).max(), 1e-30)
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= norm_bar, f"{what}: normwise relative error {rel:.3g}"
    assert err.max() <= max_bar * scale, f"{what}: max error {err.max():.3g} (max|ref| {scale:.3g})"


def compare(x, g, scale, mode, dtype, what):
    (dq, dk, dv, dk0, dv0), gq = run(x, g, scale, mode)
    ref = oracle.backward(x["q"], x["k"], x["v"], gq.float(), x["k0"], x["v0"], scale=scale,
                          mode=mode)
    check(dq, ref["dq"], dtype, what + " dq")
    check(dk, ref["dk"], dtype, what + " dk")
    check(dv, ref["dv"], dtype, what + " dv")
    if mode == oracle.GIVEN:
        check(dk0, ref["dk0"], dtype, what + " dk0")
        check(dv0, ref["dv0"], dtype, what + " dv0")
    else:
        assert dk0 is None and dv0 is None


def upstream(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed))


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B,H,T,d", [(1, 1, 1, 16), (2, 3, 37, 24), (1, 2, 130, 64)])
def test_backward_f32(mode, B, H, T, d):
    x = make_inputs(B, H, T, d, "f32", seed=100 + T + mode)
    g = upstream((B, H, T, d), 7)
    compare(x, g, 0.3, mode, "f32", f"f32 {B}x{H}x{T}x{d} mode={mode}")


@pytest.mark.parametrize("scale", [0.05, 1.0, 3.0])
def test_backward_f32_logit_ranges(scale):
    x = make_inputs(1, 2, 90, 32, "f32", seed=120)
    g = upstream((1, 2, 90, 32), 8)
    compare(x, g, scale, 2, "f32", f"f32 scale={scale}")


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("d", [64, 128, 96])
def test_backward_bf16(mode, d):
    B, H, T = 2, 2, 200
    x = make_inputs(B, H, T, d, "bf16", seed=140 + d + mode)
    g = upstream((B, H, T, d), 9)
    compare(x, g, 1.0 / d ** 0.5, mode, "bf16", f"bf16 d={d} mode={mode}")


def test_backward_empty_and_errors():
    x = make_inputs(1, 2, 8, 16, "f32", seed=150)
    dev = {k: t.cuda() for k, t in x.items()}
    o, lse = forward(dev["q"], dev["k"], dev["v"], dev["k0"], dev["v0"], mode=2)
    # empty batch in mode GIVEN: zero sink gradients
    e = {k: t[:0] for k, t in dev.items() if k not in ("k0", "v0")}
    dk0 = torch.full((2, 16), 5.0, device="cuda")
    dv0 = torch.full((2, 16), 5.0, device="cuda")
    backward(e["q"], e["k"], e["v"], o[:0], lse[:0], e["q"], dev["k0"], dev["v0"], mode=2,
             dk0=dk0, dv0=dv0)
    torch.cuda.synchronize()
    assert (dk0 == 0).all() and (dv0 == 0).all()
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(CsaError) as err:
        backward(dev["q"], dev["k"], dev["v"], o, lse, dev["q"], workspace=small)
    assert err.value.code == -1
    assert backward_workspace_bytes(1, 2, 8, 16) >= 2 * 8 * 16 * 4 * 2


@pytest.mark.parametrize("d,mode,T", [(128, 0, 700), (64, 2, 700), (128, 1, 383), (64, 0, 1000)])
def test_backward_tensor_core_tiles(d, mode, T):
    """Several key tiles (126 keys each, halo columns on both sides) and query
    tiles (128 rows), a ragged last tile, rows at every tile edge."""
    x = make_inputs(1, 2, T, d, "bf16", seed=160 + T + mode)
    g = upstream((1, 2, T, d), 10)
    compare(x, g, 1.0 / d ** 0.5, mode, "bf16", f"tc d={d} mode={mode} T={T}")


@pytest.mark.parametrize("scale", [0.02, 0.35])
def test_backward_tensor_core_logit_ranges(scale):
    # scale 0.35 at d = 64: logit gaps of several units between neighbours
    x = make_inputs(2, 2, 300, 64, "bf16", seed=170)
    g = upstream((2, 2, 300, 64), 11)
    compare(x, g, scale, 0, "bf16", f"tc scale={scale}")


def test_backward_tensor_core_matches_cuda_core_path():
    """Tensors offset by one element (2-byte aligned only) take the CUDA-core
    path; the default 16-byte aligned ones the tensor-core path.  Both are
    held to the oracle's bar here, and they must agree with each other."""
    B, H, T, d = 1, 2, 260, 64
    x = make_inputs(B, H, T, d, "bf16", seed=180)
    g = upstream((B, H, T, d), 12).to(torch.bfloat16)
    dev = {k: t.cuda() for k, t in x.items()}
    o, lse = forward(dev["q"], dev["k"], dev["v"], mode=0)
    gd = g.cuda()
    tc = backward(dev["q"], dev["k"], dev["v"], o, lse, gd, mode=0)

    def off(t):  # same values, data pointer 2 bytes past a 16-byte boundary
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
        v = buf[1:1 + t.numel()].view(t.shape)
        v.copy_(t)
        return v

    outs = [off(torch.empty_like(dev["q"])) for _ in range(3)]
    simt = backward(off(dev["q"]), off(dev["k"]), off(dev["v"]), off(o), lse, off(gd), mode=0,
                    dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    ref = oracle.backward(x["q"], x["k"], x["v"], g.float(), scale=1.0 / d ** 0.5, mode=0)
    for name, a, b in zip(("dq", "dk", "dv"), tc[:3], simt[:3]):
        check(a, ref[name], "bf16", "tensor-core " + name)
        check(b, ref[name], "bf16", "cuda-core " + name)
        diff = (a.float() - b.float()).abs().max().item()
        assert diff <= 2e-2 * np.abs(ref[name]).max(), (name, diff)


@pytest.mark.parametrize("T,d,mode", [(2048, 128, 2), (4096, 64, 0)])
def test_backward_long_rows(T, d, mode):
    """Rows of 2048 and 4096 keys: 17 and 33 key tiles per head, the lazy
    statistics of many query tiles, on two heads (the oracle runs them in
    parallel, a few seconds each)."""
    x = make_inputs(1, 2, T, d, "bf16", seed=190 + T)
    g = upstream((1, 2, T, d), 13)
    compare(x, g, 1.0 / d ** 0.5, mode, "bf16", f"long T={T} d={d}")


def test_backward_headline_shape():
    """The backward pass at the benchmark's shape (B=1, H=32, T=8192, d=128,
    zero sink, the same seeded upstream gradient), all heads in one call as
    the benchmark launches it: two scheduling groups of 16 heads, 65 key
    tiles per head.  The oracle checks the last head whole (8192 rows of dq,
    dk, dv; about 40 s of double-precision CPU work)."""
    x = workload_inputs("headline")
    B, H, T, d = x["q"].shape
    scale = 1.0 / d ** 0.5
    g = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(7))
    (dq, dk, dv, _, _), gq = run(x, g, scale, oracle.ZERO)
    h = H - 1
    sl = lambda t: t[:, h:h + 1].contiguous()
    ref = oracle.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(gq).float(), scale=scale,
                          mode=oracle.ZERO)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        check(sl(got), ref[name], "bf16", f"headline head {h} {name}")
