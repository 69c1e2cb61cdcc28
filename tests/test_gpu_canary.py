"""Output canaries: every kernel writes its outputs and nothing next to them.

Each output (o, lse, dq, dk, dv, dk0, dv0, the decode outputs) is passed as a
view into the middle of a larger buffer whose 128-byte guard regions on both
sides hold a known bit pattern.  After the call the guards must be unchanged,
and the outputs must equal those of the same call on plain tensors: bit for
bit where the kernel's order of operations is fixed, within a rounding
tolerance where it adds with reductions in no fixed order (dq, dk0, dv0).
Shapes have ragged last tiles, so the bounds checks of the last query and key
tiles are exercised at the edges of the guarded views."""
import math

import pytest
import torch

import continuous_softmax_attention_gb300 as csa
from continuous_softmax_attention_gb300.inputs import make_decode_inputs, make_inputs

pytestmark = pytest.mark.gpu

GUARD_BYTES = 128


def guarded(shape, dtype):
    """A view of the given shape inside a buffer with a guard on each side."""
    es = torch.empty((), dtype=dtype).element_size()
    g = GUARD_BYTES // es
    n = math.prod(shape)
    buf = torch.empty(g + n + g, dtype=dtype, device="cuda")
    # a fixed bit pattern in every byte of the buffer, outputs included
    buf.view(torch.uint8).fill_(0xA5)
    return buf, buf[g:g + n].view(shape), g


def guards_intact(buf, g):
    b = buf.view(torch.uint8)
    nb = g * buf.element_size()
    return bool((b[:nb] == 0xA5).all()) and bool((b[-nb:] == 0xA5).all())


@pytest.mark.parametrize("form", ["exact", "short_conv", "symmetric", "std"])
@pytest.mark.parametrize("d, T, mode, dtype", [
    (128, 300, 2, "bf16"), (128, 129, 1, "bf16"), (64, 257, 0, "bf16"), (64, 100, 2, "bf16"),
    (96, 150, 2, "bf16"),  # bf16 on the CUDA-core kernels
    (32, 70, 1, "f32"),
])
def test_forward_writes_only_its_outputs(form, d, T, mode, dtype):
    B, H = 2, 3
    x = make_inputs(B, H, T, d, dtype, seed=T + d)
    g = {k: t.cuda() for k, t in x.items()}
    scale = d ** -0.5
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ob, o, go = guarded((B, H, T, d), tdt)
    lb, lse, gl = guarded((B, H, T), torch.float32)

    def call(out, l):
        if form == "std":
            return csa.std_forward(g["q"], g["k"], g["v"], scale=scale, out=out, lse=l)
        if form == "symmetric":
            return csa.forward_symmetric(g["q"], g["k"], g["v"], scale=scale, out=out, lse=l)
        return csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale,
                           out=out, lse=l, short_conv=form == "short_conv")

    call(o, lse)
    ro, rl = call(None, None)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    assert guards_intact(ob, go) and guards_intact(lb, gl)
    assert torch.equal(o, ro) and torch.equal(lse, rl)


@pytest.mark.parametrize("d, T, mode", [(128, 300, 2), (64, 257, 1)])
def test_backward_writes_only_its_outputs(d, T, mode):
    B, H = 2, 2
    x = make_inputs(B, H, T, d, "bf16", seed=5 + T)
    g = {k: t.cuda() for k, t in x.items()}
    scale = d ** -0.5
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale)
    gen = torch.Generator().manual_seed(9)
    dout = torch.randn(B, H, T, d, generator=gen).to(torch.bfloat16).cuda()
    bufs = {n: guarded((B, H, T, d), torch.bfloat16) for n in ("dq", "dk", "dv")}
    bufs.update({n: guarded((H, d), torch.float32) for n in ("dk0", "dv0")})
    kw = {n: v[1] for n, v in bufs.items()}
    if mode != 2:
        kw.pop("dk0")
        kw.pop("dv0")
    got = csa.backward(g["q"], g["k"], g["v"], o, lse, dout, g["k0"], g["v0"], mode=mode,
                       scale=scale, **kw)
    ref = csa.backward(g["q"], g["k"], g["v"], o, lse, dout, g["k0"], g["v0"], mode=mode,
                       scale=scale)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    for n, (buf, _, gg) in bufs.items():
        assert guards_intact(buf, gg), n
    names = ("dq", "dk", "dv", "dk0", "dv0")
    for n, a, b in zip(names, got, ref):
        if a is None:
            assert b is None and mode != 2
            continue
        if n in ("dk", "dv"):
            assert torch.equal(a, b), n
        else:  # summed by reductions in no fixed order
            af, bf = a.float(), b.float()
            tol = 2 ** -7 * max(bf.abs().max().item(), 1e-6) if n == "dq" else 1e-5 * max(
                bf.abs().max().item(), 1e-6)
            assert (af - bf).abs().max().item() <= tol, n


@pytest.mark.parametrize("d, T", [(128, 700), (64, 300)])
def test_decode_writes_only_its_outputs(d, T):
    B, H = 3, 2
    x = make_decode_inputs(B, H, T, d, seed=11, len_lo=1)
    g = {k: t.cuda() for k, t in x.items() if k != "seqlens"}
    sl = torch.as_tensor(x["seqlens"], dtype=torch.int32).cuda()
    ob, o, go = guarded((B, H, d), torch.bfloat16)
    lb, lse, gl = guarded((B, H), torch.float32)
    csa.decode(g["q"], g["k"], g["v"], g["k0"], g["v0"], seqlens=sl, mode=2, out=o, lse=lse)
    ro, rl = csa.decode(g["q"], g["k"], g["v"], g["k0"], g["v0"], seqlens=sl, mode=2)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    assert guards_intact(ob, go) and guards_intact(lb, gl)
    assert torch.equal(o, ro) and torch.equal(lse, rl)
