"""Multi-GPU use of the forward pass: one process per GPU, no collective on
the data path.

The (b, h) problems of a batch are independent (each head's rows attend
only its own keys), so N ranks split the B*H problems into contiguous
shards, each runs the CUDA kernel on its shard, and an all-gather assembles
the result where the caller wants it in one place.  The only collectives are
that optional gather, a barrier and the max of timings in the benchmark.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def head_shard(n_problems: int, world: int, rank: int):
    """Contiguous, balanced [start, stop) of the flattened (b, h) problems."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(n_problems, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def shard_inputs(q, k, v, k0, v0, world: int, rank: int):
    """This rank's problems as a [1, n, T, d] batch (views of q, k, v) and,
    for the per-head sink pair, the matching [n, d] rows of k0 and v0."""
    B, H, T, d = q.shape
    start, stop = head_shard(B * H, world, rank)
    flat = lambda t: t.reshape(B * H, T, d)[start:stop].unsqueeze(0)
    heads = torch.arange(start, stop, device=q.device) % H
    k0s = k0.index_select(0, heads) if k0 is not None else None
    v0s = v0.index_select(0, heads) if v0 is not None else None
    return flat(q), flat(k), flat(v), k0s, v0s, (start, stop)


def gather_outputs(o_s, lse_s, B: int, H: int, world: int, group=None):
    """All-gather of the shards of every rank into full [B, H, T, d] and
    [B, H, T] tensors (shards padded to the largest size for the exchange)."""
    _, n, T, d = o_s.shape
    sizes = [head_shard(B * H, world, r) for r in range(world)]
    width = max(b - a for a, b in sizes)
    pad_o = torch.zeros((width, T, d), dtype=o_s.dtype, device=o_s.device)
    pad_l = torch.zeros((width, T), dtype=lse_s.dtype, device=lse_s.device)
    pad_o[:n] = o_s[0]
    pad_l[:n] = lse_s[0]
    go = [torch.empty_like(pad_o) for _ in range(world)]
    gl = [torch.empty_like(pad_l) for _ in range(world)]
    dist.all_gather(go, pad_o, group=group)
    dist.all_gather(gl, pad_l, group=group)
    o = torch.cat([go[r][: b - a] for r, (a, b) in enumerate(sizes)]).reshape(B, H, T, d)
    lse = torch.cat([gl[r][: b - a] for r, (a, b) in enumerate(sizes)]).reshape(B, H, T)
    return o, lse


def forward_sharded(q, k, v, k0=None, v0=None, *, mode: int = 0, scale=None, gather=True,
                    group=None, fn=None):
    """Runs the forward pass on this rank's share of the (b, h) problems.

    fn(q, k, v, k0, v0, mode=, scale=) -> (o, lse) computes one shard; it is
    the CUDA kernel (continuous_softmax_attention_gb300.forward) by default.
    Returns the full (o, lse) when gather is true, else this rank's shard and
    its [start, stop) range."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if fn is None:
        from . import forward as fn
    qs, ks, vs, k0s, v0s, rng = shard_inputs(q, k, v, k0, v0, world, rank)
    o_s, lse_s = fn(qs.contiguous(), ks.contiguous(), vs.contiguous(), k0s, v0s, mode=mode,
                    scale=scale)
    if not gather or world == 1:
        return (o_s, lse_s) if gather else (o_s, lse_s, rng)
    B, H = q.shape[0], q.shape[1]
    return gather_outputs(o_s, lse_s, B, H, world, group)


def max_over_ranks(value: float, device=None, group=None) -> float:
    """The largest value over all ranks (the benchmark's timed region)."""
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def backward_sharded(q, k, v, out, lse, dout, k0=None, v0=None, *, mode: int = 0, scale=None,
                     gather=True, group=None, fn=None):
    """The backward pass on this rank's share of the (b, h) problems.

    fn(q, k, v, out, lse, dout, k0, v0, mode=, scale=) -> (dq, dk, dv, dk0,
    dv0) computes one shard (the CUDA kernel, continuous_softmax_attention_
    gb300.backward, by default).  dq, dk, dv need no exchange; the gradients
    of the per-head sink pair (mode GIVEN) sum over the whole batch, so each
    rank's partial [H, d] sums are all-reduced.  Returns (dq, dk, dv, dk0,
    dv0) for the full problem when gather is true, else this rank's dq, dk,
    dv shard with the all-reduced dk0, dv0 and its [start, stop) range."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if fn is None:
        from . import backward as fn
    B, H, T, d = q.shape
    start, stop = head_shard(B * H, world, rank)
    flat = lambda t: t.reshape(B * H, T, d)[start:stop].unsqueeze(0).contiguous()
    lse_s = lse.reshape(B * H, T)[start:stop].unsqueeze(0).contiguous()
    heads = torch.arange(start, stop, device=q.device) % H
    k0s = k0.index_select(0, heads) if (k0 is not None and mode == 2) else None
    v0s = v0.index_select(0, heads) if (v0 is not None and mode == 2) else None
    dq, dk, dv, dk0_s, dv0_s = fn(flat(q), flat(k), flat(v), flat(out), lse_s, flat(dout), k0s,
                                  v0s, mode=mode, scale=scale)
    dk0 = dv0 = None
    if mode == 2:
        # the shard's problems are [1, n] with head ids `heads`: fold its
        # per-problem sink gradients back onto the H heads, then sum ranks
        dk0 = torch.zeros((H, d), dtype=torch.float64, device=q.device)
        dv0 = torch.zeros((H, d), dtype=torch.float64, device=q.device)
        dk0.index_add_(0, heads, dk0_s.to(torch.float64))
        dv0.index_add_(0, heads, dv0_s.to(torch.float64))
        if world > 1:
            dist.all_reduce(dk0, group=group)
            dist.all_reduce(dv0, group=group)
    if not gather:
        return dq, dk, dv, dk0, dv0, (start, stop)
    if world == 1:
        return (dq.reshape(B, H, T, d), dk.reshape(B, H, T, d), dv.reshape(B, H, T, d), dk0, dv0)
    lse_dummy = torch.zeros(dq.shape[:-1], dtype=torch.float32, device=q.device)
    gq, _ = gather_outputs(dq, lse_dummy, B, H, world, group)
    gk, _ = gather_outputs(dk, lse_dummy, B, H, world, group)
    gv, _ = gather_outputs(dv, lse_dummy, B, H, world, group)
    return gq, gk, gv, dk0, dv0


def decode_sharded(q, k_cache, v_cache, k0=None, v0=None, *, seqlens=None, mode: int = 0,
                   scale=None, gather=True, group=None, fn=None):
    """A decode step on this rank's share of the sequences (whole sequences
    per rank, so each keeps its own length).  fn(q, k, v, k0, v0, seqlens=,
    mode=, scale=) -> (o, lse) computes one shard (the CUDA decode step by
    default).  No collective on the data path; gather=True all-gathers the
    per-sequence outputs."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if fn is None:
        from . import decode as fn
    B = k_cache.shape[0]
    start, stop = head_shard(B, world, rank)
    sl = None if seqlens is None else seqlens[start:stop].contiguous()
    o, lse = fn(q[start:stop].contiguous(), k_cache[start:stop].contiguous(),
                v_cache[start:stop].contiguous(), k0, v0, seqlens=sl, mode=mode, scale=scale)
    if not gather or world == 1:
        return (o, lse) if gather else (o, lse, (start, stop))
    H, d = q.shape[1], q.shape[2]
    width = max(b - a for a, b in (head_shard(B, world, r) for r in range(world)))
    pad_o = torch.zeros((width, H, d), dtype=o.dtype, device=o.device)
    pad_l = torch.zeros((width, H), dtype=lse.dtype, device=lse.device)
    pad_o[:stop - start] = o
    pad_l[:stop - start] = lse
    go = [torch.empty_like(pad_o) for _ in range(world)]
    gl = [torch.empty_like(pad_l) for _ in range(world)]
    dist.all_gather(go, pad_o, group=group)
    dist.all_gather(gl, pad_l, group=group)
    sizes = [head_shard(B, world, r) for r in range(world)]
    o_full = torch.cat([go[r][: b - a] for r, (a, b) in enumerate(sizes)])
    l_full = torch.cat([gl[r][: b - a] for r, (a, b) in enumerate(sizes)])
    return o_full, l_full


# ---------------------------------------------------------------- context parallelism
# One long sequence's KV cache split along its time axis: rank r owns the
# positions [lo_r, hi_r) of every row (position 0 the sink, position i >= 1
# cache row i - 1) and holds those cache rows plus one neighbour on each
# side, which the correction b of its first and last positions needs.  Each
# rank computes the partial (o_r, lse_r) of its positions; one all-gather and
# an lse-weighted merge give the whole row's result.  This is the only
# exchange step of the decode path.


def context_ranges(T: int, world: int):
    """Contiguous, balanced ranges [lo, hi) partitioning the positions 0..T
    over `world` ranks.  No range starts at position 1 (right after the
    sink), so a cut that would fall there moves to 2; every range is
    non-empty, which needs T + 1 >= 2 * world."""
    if world < 1 or T + 1 < 2 * world:
        raise ValueError("need T + 1 >= 2 * world positions")
    cuts = [0]
    for r in range(1, world):
        c = (r * (T + 1)) // world
        cuts.append(max(c, cuts[-1] + 1, 2))
    cuts.append(T + 1)
    for a, b in zip(cuts, cuts[1:]):
        if b <= a:
            raise ValueError("positions too few for the ranks")
    return list(zip(cuts[:-1], cuts[1:]))


def cache_shard(k_cache, v_cache, pos_lo: int, pos_hi: int):
    """The cache rows a range's rank holds: [max(pos_lo - 2, 0), min(pos_hi, T))."""
    T = k_cache.shape[2]
    r0, r1 = max(pos_lo - 2, 0), min(pos_hi, T)
    return k_cache[:, :, r0:r1].contiguous(), v_cache[:, :, r0:r1].contiguous()


def gather_parts(o_r, lse_r, group=None):
    """All-gather of every rank's partial: ([R, B, H, d], [R, B, H])."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        return o_r.unsqueeze(0), lse_r.unsqueeze(0)
    go = [torch.empty_like(o_r) for _ in range(world)]
    gl = [torch.empty_like(lse_r) for _ in range(world)]
    dist.all_gather(go, o_r.contiguous(), group=group)
    dist.all_gather(gl, lse_r.contiguous(), group=group)
    return torch.stack(go), torch.stack(gl)


def decode_context_parallel(q, k_shard, v_shard, T: int, k0=None, v0=None, *, seqlens=None,
                            mode: int = 0, scale=None, group=None, fn=None, merge_fn=None):
    """A decode step with the cache split along time across the ranks of
    `group` (context_ranges(T, world)[rank] is this rank's range, k_shard and
    v_shard its cache_shard).  fn computes the partial of this rank's
    positions (the CUDA csa_decode_range by default), merge_fn merges the
    gathered partials (csa_decode_merge_ranges by default).  Every rank gets
    the whole result (o, lse)."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    lo, hi = context_ranges(T, world)[rank]
    if fn is None:
        from . import decode_range as fn
    if merge_fn is None:
        from . import decode_merge_ranges as merge_fn
    o_r, lse_r = fn(q, k_shard, v_shard, T, lo, hi, k0, v0, seqlens=seqlens, mode=mode,
                    scale=scale)
    o_parts, lse_parts = gather_parts(o_r, lse_r, group)
    return merge_fn(o_parts, lse_parts)
