"""The multi-rank paths with the CUDA kernels in every rank: two processes
on one GPU, with gloo carrying CPU copies for the exchange.  The (b, h)
shards of the forward and backward must give one process's result (bit for
bit where the kernels are deterministic), and a decode with each cache split
along time over the ranks must give the same ranges run in one process.  The
ranks' kernels are independent launches that never wait on one another; only
the host-side gathers and the all-reduce of the sink gradients cross ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

B, H, T, D = 2, 3, 700, 64  # 6 problems: 3 per rank
SCALE = 0.125


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from continuous_softmax_attention_gb300.inputs import make_inputs

    x = make_inputs(B, H, T, D, "bf16", seed=11)
    g = torch.randn(B, H, T, D, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    return x, g


def _worker(rank, world, port, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import continuous_softmax_attention_gb300 as csa
        from continuous_softmax_attention_gb300.dist import backward_sharded, forward_sharded

        x, g = _inputs()
        dev = torch.device("cuda:0")

        def fwd(q_, k_, v_, k0_, v0_, mode, scale):
            on = lambda t: None if t is None else t.to(dev)
            o, lse = csa.forward(on(q_), on(k_), on(v_), on(k0_), on(v0_), mode=mode, scale=scale)
            return o.cpu(), lse.cpu()

        def bwd(q_, k_, v_, o_, lse_, dout_, k0_, v0_, mode, scale):
            on = lambda t: None if t is None else t.to(dev)
            r = csa.backward(on(q_), on(k_), on(v_), on(o_), on(lse_), on(dout_), on(k0_), on(v0_),
                             mode=mode, scale=scale)
            return tuple(None if t is None else t.float().cpu() for t in r)

        o, lse = forward_sharded(x["q"], x["k"], x["v"], x["k0"], x["v0"], mode=mode, scale=SCALE,
                                 fn=fwd)
        grads = backward_sharded(x["q"], x["k"], x["v"], o, lse, g, x["k0"], x["v0"], mode=mode,
                                 scale=SCALE, fn=bwd)
        st = csa.device_status()
        if rank == 0:
            q.put((o, lse, grads, st))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", [0, 2])
def test_two_ranks_on_the_kernels_match_one_process(mode):
    import continuous_softmax_attention_gb300 as csa

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    o, lse, grads, st = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert st == 0
    x, g = _inputs()
    dev = torch.device("cuda:0")
    k0 = x["k0"].to(dev) if mode == 2 else None
    v0 = x["v0"].to(dev) if mode == 2 else None
    ro, rl = csa.forward(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), k0, v0, mode=mode,
                         scale=SCALE)
    assert torch.equal(o, ro.cpu()) and torch.equal(lse, rl.cpu())
    ref = csa.backward(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), ro, rl, g.to(dev), k0, v0,
                       mode=mode, scale=SCALE)
    torch.cuda.synchronize()
    # dk, dv: accumulated per key tile in a fixed order, the same bits
    for name, a, b in zip(("dk", "dv"), grads[1:3], ref[1:3]):
        assert torch.equal(a, b.float().cpu()), name
    # dq: the key tiles add their parts into fp32 in whatever order they
    # finish, so two launches may round differently in the last bf16 bit
    dq, rdq = grads[0], ref[0].float().cpu()
    assert (dq - rdq).abs().max() <= 2e-2 * rdq.abs().max(), "dq"
    if mode == 2:
        # the sink gradients are sums over the batch: two ranks' partial
        # sums added by the all-reduce, against one kernel's accumulation
        for name, a, b in zip(("dk0", "dv0"), grads[3:], ref[3:]):
            a, b = a.float(), b.float().cpu()
            assert (a - b).abs().max() <= 1e-3 * b.abs().max(), name


def _cp_worker(rank, world, port, T, d, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import continuous_softmax_attention_gb300 as csa
        from continuous_softmax_attention_gb300.dist import (cache_shard, context_ranges,
                                                             decode_context_parallel)
        from continuous_softmax_attention_gb300.inputs import make_decode_inputs

        dev = torch.device("cuda:0")
        x = make_decode_inputs(4, 2, T, d, 71 + mode, 1)
        sl = torch.tensor([T, 1, T // 2, T - 5], dtype=torch.int32)
        lo, hi = context_ranges(T, world)[rank]
        ks, vs = cache_shard(x["k"], x["v"], lo, hi)
        on = lambda t: None if t is None else t.to(dev)

        def part(q_, k_, v_, T_, lo_, hi_, k0_, v0_, seqlens, mode, scale):
            o, lse = csa.decode_range(on(q_), on(k_), on(v_), T_, lo_, hi_, on(k0_), on(v0_),
                                      seqlens=on(seqlens), mode=mode, scale=scale)
            return o.cpu(), lse.cpu()

        def merge(o_parts, lse_parts):
            o, lse = csa.decode_merge_ranges(on(o_parts), on(lse_parts))
            return o.cpu(), lse.cpu()

        o, lse = decode_context_parallel(x["q"], ks, vs, T, x["k0"], x["v0"], seqlens=sl,
                                         mode=mode, scale=d ** -0.5, fn=part, merge_fn=merge)
        if rank == 0:
            q.put((o, lse, csa.device_status()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", [1, 2])
def test_context_parallel_decode_on_the_kernels_matches_one_process(mode):
    """The cache of each sequence split along time over two processes, each
    running csa_decode_range on its shard; the gathered partials merged by
    csa_decode_merge_ranges equal the same ranges run in one process."""
    import continuous_softmax_attention_gb300 as csa
    from continuous_softmax_attention_gb300.dist import cache_shard, context_ranges
    from continuous_softmax_attention_gb300.inputs import make_decode_inputs

    world, T, d = 2, 900, 128
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, world, port, T, d, mode, q))
             for r in range(world)]
    for p in procs:
        p.start()
    o, lse, st = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert st == 0
    dev = torch.device("cuda:0")
    x = make_decode_inputs(4, 2, T, d, 71 + mode, 1)
    sl = torch.tensor([T, 1, T // 2, T - 5], dtype=torch.int32, device=dev)
    g = {k: t.to(dev) for k, t in x.items() if k != "seqlens"}
    parts = []
    for lo, hi in context_ranges(T, world):
        ks, vs = cache_shard(g["k"], g["v"], lo, hi)
        parts.append(csa.decode_range(g["q"], ks, vs, T, lo, hi, g["k0"], g["v0"], seqlens=sl,
                                      mode=mode, scale=d ** -0.5))
    ro, rl = csa.decode_merge_ranges(torch.stack([a for a, _ in parts]),
                                     torch.stack([b for _, b in parts]))
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu()) and torch.equal(lse, rl.cpu())
