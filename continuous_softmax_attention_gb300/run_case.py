"""Runs the kernels a few times at one shape (for profilers).

    python -m continuous_softmax_attention_gb300.run_case --B 1 --H 24 --T 8192 --d 128
    python -m continuous_softmax_attention_gb300.run_case --decode --B 4 --H 32 --T 8192

Inputs come from the seeded generator; each iteration launches the
continuous kernel once and, unless --no-std, the standard kernel once.
With --decode each iteration is one decode step (lengths drawn from
[T/2, T]); with --backward one forward pass, then each iteration is one
backward pass.
"""
from __future__ import annotations

import argparse
import math

import torch

import continuous_softmax_attention_gb300 as csa
from continuous_softmax_attention_gb300.inputs import make_inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=24)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--mode", type=int, default=0)
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--no-std", action="store_true")
    ap.add_argument("--decode", action="store_true")
    ap.add_argument("--backward", action="store_true")
    ap.add_argument("--short-conv", action="store_true",
                    help="the first-order (eq. (13)) form instead of the exact one")
    ap.add_argument("--log-domain", action="store_true",
                    help="the exact form's weights formed in the log domain")
    a = ap.parse_args()
    if a.decode:
        return run_decode(a)
    if a.backward:
        return run_backward(a)
    x = make_inputs(a.B, a.H, a.T, a.d, "bf16", seed=0)
    g = {k: v.cuda() for k, v in x.items()}
    scale = 1.0 / math.sqrt(a.d)
    for _ in range(a.iters):
        o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=a.mode, scale=scale,
                             short_conv=a.short_conv, log_domain=a.log_domain)
        if not a.no_std:
            csa.std_forward(g["q"], g["k"], g["v"], scale=scale)
    torch.cuda.synchronize()
    st = csa.device_status()
    print(f"ok status={st} o_mean={o.float().abs().mean().item():.5f}")
    if st != 0:
        raise SystemExit(1)


def run_backward(a):
    x = make_inputs(a.B, a.H, a.T, a.d, "bf16", seed=0)
    g = {k: v.cuda() for k, v in x.items()}
    scale = 1.0 / math.sqrt(a.d)
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=a.mode, scale=scale)
    dout = torch.randn(a.B, a.H, a.T, a.d, generator=torch.Generator().manual_seed(1))
    dout = dout.to(torch.bfloat16).cuda()
    for _ in range(a.iters):
        dq, dk, dv, _, _ = csa.backward(g["q"], g["k"], g["v"], o, lse, dout, g["k0"], g["v0"],
                                        mode=a.mode, scale=scale)
    torch.cuda.synchronize()
    st = csa.device_status()
    print(f"ok status={st} dq_mean={dq.float().abs().mean().item():.5f}")
    if st != 0:
        raise SystemExit(1)


def run_decode(a):
    from continuous_softmax_attention_gb300.inputs import make_decode_inputs

    x = make_decode_inputs(a.B, a.H, a.T, a.d, seed=0, len_lo=max(1, a.T // 2))
    g = {k: v.cuda() for k, v in x.items()}
    for _ in range(a.iters):
        o, lse = csa.decode(g["q"], g["k"], g["v"], g["k0"], g["v0"], seqlens=g["seqlens"],
                            mode=a.mode)
    torch.cuda.synchronize()
    st = csa.device_status()
    print(f"ok status={st} o_mean={o.float().abs().mean().item():.5f}")
    if st != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
