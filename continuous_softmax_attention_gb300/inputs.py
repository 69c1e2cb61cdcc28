"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the attention method: it only draws
Gaussian tensors, optionally rotates q and k with RoPE (input preparation for
the mid-size training shape), and rounds to the storage dtype.  Both the CUDA
path and the CPU oracle consume exactly the tensors it returns.

Recipe (every workload): a CPU ``torch.Generator`` seeded with the workload's
seed draws q, k, v (each [B, H, T, d]) and then k0, v0 (each [H, d]) from
N(0, 1) in float32, in that order.  RoPE, when asked for, rotates the pairs
(i, i + d/2) of q and k by the angle pos * 10000^(-2i/d) at positions
0..T-1, in float32.  The result is rounded to bf16 (round to nearest even)
when the dtype is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

ZERO, COPY_FIRST, GIVEN = 0, 1, 2
MODE_NAMES = {ZERO: "zero", COPY_FIRST: "copy_first", GIVEN: "given"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str  # "f32" or "bf16"
    seed: int
    scales: tuple = ()  # empty -> 1/sqrt(d)
    modes: tuple = (ZERO,)
    rope: bool = False
    notes: str = ""

    def scale_list(self):
        return list(self.scales) if self.scales else [1.0 / math.sqrt(self.d)]


# The five workloads of the method's evaluation plan (all synthetic).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 64, 16, "f32", 0, (0.25,), (ZERO,),
                     notes="fp32, also checked by quadrature of eq. (2)"),
    "stress": Workload("stress", 2, 4, 512, 64, "bf16", 1, (0.125, 1.0, 4.0), (ZERO, COPY_FIRST),
                       notes="logit gaps up to ~+-200 at scale 4"),
    "mid": Workload("mid", 4, 16, 2048, 128, "bf16", 2, (), (ZERO,), rope=True,
                    notes="RoPE base 10000 applied to q, k"),
    "headline": Workload("headline", 1, 32, 8192, 128, "bf16", 3, (), (ZERO,),
                         notes="timed next to standard causal attention"),
    "long": Workload("long", 1, 8, 32768, 64, "bf16", 4, (), (GIVEN,),
                     notes="per-head k0, v0 ~ N(0,1)"),
}


def rope(x: torch.Tensor, base: float = 10000.0) -> torch.Tensor:
    """Rotate-half RoPE on the last dim of a float32 [..., T, d] tensor."""
    T, d = x.shape[-2], x.shape[-1]
    half = d // 2
    inv = base ** (-torch.arange(0, half, dtype=torch.float64) * 2.0 / d)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
    cos = torch.cos(ang).float()
    sin = torch.sin(ang).float()
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x1 * sin + x2 * cos], dim=-1)


def make_inputs(B, H, T, d, dtype="bf16", seed=0, rope_qk=False):
    """Returns dict(q, k, v, k0, v0) of CPU tensors in the storage dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
    k0 = torch.randn(H, d, generator=g, dtype=torch.float32)
    v0 = torch.randn(H, d, generator=g, dtype=torch.float32)
    if rope_qk:
        q, k = rope(q), rope(k)
    if dtype == "bf16":
        cast = lambda t: t.to(torch.bfloat16)
    elif dtype == "f32":
        cast = lambda t: t.contiguous()
    else:
        raise ValueError(f"dtype {dtype!r}")
    return {"q": cast(q), "k": cast(k), "v": cast(v), "k0": cast(k0), "v0": cast(v0)}


def workload_inputs(name: str):
    w = WORKLOADS[name]
    return make_inputs(w.B, w.H, w.T, w.d, w.dtype, w.seed, w.rope)


def algorithmic_flops(B, H, T, d, continuous=True):
    """Matmul flops the method must do: 4*d per (query, key) pair.

    A continuous row t = r+1 has t+1 pairs (the sink included); a standard
    row has t pairs."""
    pairs = B * H * (T * (T + 3) // 2 if continuous else T * (T + 1) // 2)
    return 4 * d * pairs


# Decode step: the newest token of each of B sequences against its KV cache.
# Recipe: a CPU generator seeded with `seed` draws q [B, H, d], k, v
# [B, H, T, d], k0, v0 [H, d] from N(0, 1) in float32, in that order, then the
# lengths n_b uniformly from the integers [len_lo, T]; tensors are rounded to
# bf16.  Rows past n_b of the cache are drawn too (they are never read).
@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    T: int
    d: int
    seed: int
    len_lo: int
    mode: int = ZERO
    notes: str = ""


DECODE_WORKLOADS = {
    "decode_small": DecodeWorkload("decode_small", 3, 2, 700, 128, 5, 1,
                                   notes="parity case: several chunks and a ragged tail"),
    "decode": DecodeWorkload("decode", 16, 32, 8192, 128, 6, 4096,
                             notes="headline head shape, 16 sequences, lengths in [T/2, T]"),
}


def make_decode_inputs(B, H, T, d, seed=0, len_lo=1):
    """Returns dict(q, k, v, k0, v0, seqlens) of CPU tensors (bf16, int32)."""
    if not 1 <= len_lo <= T:
        raise ValueError("need 1 <= len_lo <= T")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    bf = lambda *shape: torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    q = bf(B, H, d)
    k = torch.empty(B, H, T, d, dtype=torch.bfloat16)
    v = torch.empty(B, H, T, d, dtype=torch.bfloat16)
    for t in (k, v):  # one sequence at a time keeps the float32 staging small
        for b in range(B):
            t[b] = torch.randn(H, T, d, generator=g, dtype=torch.float32)
    k0, v0 = bf(H, d), bf(H, d)
    seqlens = torch.randint(len_lo, T + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return {"q": q, "k": k, "v": v, "k0": k0, "v0": v0, "seqlens": seqlens}


def decode_workload_inputs(name: str):
    w = DECODE_WORKLOADS[name]
    return make_decode_inputs(w.B, w.H, w.T, w.d, w.seed, w.len_lo)


def decode_bytes(seqlens, H, d):
    """HBM bytes a decode step must move: every used cached key and value
    row once (bf16), the queries and outputs (bf16) and lse (fp32)."""
    n = int(sum(int(x) for x in seqlens))
    B = len(seqlens)
    return 2 * n * H * d * 2 + 2 * B * H * d * 2 + B * H * 4
