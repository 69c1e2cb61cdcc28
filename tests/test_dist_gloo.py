"""The multi-rank path on CPU: two gloo ranks split the (b, h) problems,
compute their shards (with the CPU oracle standing in for the GPU kernel,
which these CPU tests do not launch), gather them, and must reproduce the
single-process result exactly; the benchmark's max-over-ranks reduction is
checked too."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from continuous_softmax_attention_gb300.dist import (forward_sharded, head_shard, max_over_ranks)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fn(q, k, v, k0, v0, mode, scale):
    import oracle

    o, lse = oracle.forward(q, k, v, k0, v0, scale=scale, mode=mode, nthreads=1)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _worker(rank, world, port, B, H, T, d, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from continuous_softmax_attention_gb300.inputs import make_inputs

        x = make_inputs(B, H, T, d, "f32", seed=42)
        o, lse = forward_sharded(x["q"], x["k"], x["v"], x["k0"], x["v0"], mode=mode, scale=0.4,
                                 fn=_oracle_fn)
        t = max_over_ranks(10.0 + rank)
        if rank == 0:
            q.put((o.numpy(), lse.numpy(), t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B,H,mode,world", [(2, 3, 2, 2), (1, 5, 0, 2), (3, 1, 1, 2), (2, 3, 2, 4),
                                            (1, 3, 0, 4)])
def test_gloo_ranks_match_single_process(B, H, mode, world):
    """world ranks each take a shard of the B*H problems (with 3 problems
    over 4 ranks, one rank has none) and the gathered result equals one
    process's."""
    import oracle
    from continuous_softmax_attention_gb300.inputs import make_inputs

    T, d = 40, 8
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, B, H, T, d, mode, q))
             for r in range(world)]
    for p in procs:
        p.start()
    o, lse, t = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = make_inputs(B, H, T, d, "f32", seed=42)
    ro, rl = oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=0.4, mode=mode)
    assert np.array_equal(o, ro) and np.array_equal(lse, rl)
    assert t == 10.0 + world - 1  # the max over ranks of 10 + rank


def test_head_shard_partition():
    for n in (0, 1, 5, 32, 33):
        for world in (1, 2, 3, 8):
            got = [head_shard(n, world, r) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
            sizes = [b - a for a, b in got]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_shard(4, 2, 2)


def test_single_process_path():
    from continuous_softmax_attention_gb300.inputs import make_inputs

    x = make_inputs(1, 2, 10, 4, "f32", seed=1)
    o, lse = forward_sharded(x["q"], x["k"], x["v"], x["k0"], x["v0"], mode=2, scale=0.3,
                             fn=_oracle_fn)
    assert o.shape == (1, 2, 10, 4) and lse.shape == (1, 2, 10)
    assert max_over_ranks(3.5) == 3.5


def _oracle_bwd(q, k, v, out, lse, dout, k0, v0, mode, scale):
    import oracle

    r = oracle.backward(q, k, v, dout, k0, v0, scale=scale, mode=mode, nthreads=1)
    t = lambda a: None if a is None else torch.from_numpy(a)
    return t(r["dq"]), t(r["dk"]), t(r["dv"]), t(r["dk0"]), t(r["dv0"])


def _bwd_worker(rank, world, port, B, H, T, d, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from continuous_softmax_attention_gb300.dist import backward_sharded
        from continuous_softmax_attention_gb300.inputs import make_inputs

        x = make_inputs(B, H, T, d, "f32", seed=43)
        g = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(2))
        lse = torch.zeros(B, H, T)
        res = backward_sharded(x["q"], x["k"], x["v"], x["q"], lse, g, x["k0"], x["v0"],
                               mode=mode, scale=0.5, fn=_oracle_bwd)
        if rank == 0:
            q.put(tuple(None if t is None else t.numpy() for t in res))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B,H,mode,world", [(2, 3, 2, 2), (1, 3, 0, 2), (3, 1, 1, 2), (1, 3, 2, 4)])
def test_backward_gloo_ranks(B, H, mode, world):
    """dq, dk, dv shard with no exchange; the sink gradients (mode GIVEN) are
    all-reduced across ranks, one of which may hold no problems; everything
    matches one process."""
    import oracle
    from continuous_softmax_attention_gb300.inputs import make_inputs

    T, d = 12, 4
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, world, port, B, H, T, d, mode, q))
             for r in range(world)]
    for p in procs:
        p.start()
    dq, dk, dv, dk0, dv0 = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = make_inputs(B, H, T, d, "f32", seed=43)
    g = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(2))
    ref = oracle.backward(x["q"], x["k"], x["v"], g, x["k0"], x["v0"], scale=0.5, mode=mode)
    assert np.array_equal(dq, ref["dq"]) and np.array_equal(dk, ref["dk"])
    assert np.array_equal(dv, ref["dv"])
    if mode == 2:
        assert np.abs(dk0 - ref["dk0"]).max() < 1e-12 and np.abs(dv0 - ref["dv0"]).max() < 1e-12
    else:
        assert dk0 is None and dv0 is None


def _oracle_decode(q, k, v, k0, v0, seqlens, mode, scale):
    """Row n_b - 1 of eq. (8) for every (b, h): the decode result."""
    import oracle

    B, H, T, d = k.shape
    o = torch.zeros(B, H, d, dtype=torch.float64)
    lse = torch.zeros(B, H, dtype=torch.float64)
    for b in range(B):
        n = int(seqlens[b])
        qf = torch.zeros(1, H, n, d)
        qf[0, :, n - 1] = q[b]
        ro, rl = oracle.forward_rows(qf, k[b:b + 1, :, :n], v[b:b + 1, :, :n],
                                     oracle.flat_rows(1, H, n, [(0, h, n - 1) for h in range(H)]),
                                     k0, v0, scale=scale, mode=mode, nthreads=1)
        o[b] = torch.from_numpy(ro)
        lse[b] = torch.from_numpy(rl)
    return o, lse


def _dec_worker(rank, world, port, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from continuous_softmax_attention_gb300.dist import decode_sharded
        from continuous_softmax_attention_gb300.inputs import make_decode_inputs

        x = make_decode_inputs(5, 2, 30, 8, seed=8, len_lo=1)
        o, lse = decode_sharded(x["q"].float(), x["k"].float(), x["v"].float(), x["k0"].float(),
                                x["v0"].float(), seqlens=x["seqlens"], mode=mode, scale=0.4,
                                fn=lambda *a, seqlens, mode, scale: _oracle_decode(
                                    *a, seqlens, mode, scale))
        if rank == 0:
            q.put((o.numpy(), lse.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", [0, 2])
def test_decode_two_gloo_ranks(mode):
    """Whole sequences per rank, no collective on the data path; the gathered
    step equals one process's."""
    from continuous_softmax_attention_gb300.inputs import make_decode_inputs

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dec_worker, args=(r, 2, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    o, lse = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = make_decode_inputs(5, 2, 30, 8, seed=8, len_lo=1)
    ro, rl = _oracle_decode(x["q"].float(), x["k"].float(), x["v"].float(), x["k0"].float(),
                            x["v0"].float(), x["seqlens"], mode, 0.4)
    assert np.array_equal(o, ro.numpy()) and np.array_equal(lse, rl.numpy())


# ---------------------------------------------------------------- context parallelism
def _merge_np(o_parts, lse_parts):
    """lse-weighted merge of range partials (test-side, float64)."""
    lses = lse_parts.double()
    L = lses.max(dim=0).values
    w = torch.exp(lses - L)
    o = (w[..., None] * o_parts.double()).sum(dim=0) / w.sum(dim=0)[..., None]
    return o, L + torch.log(w.sum(dim=0))


def _cp_worker(rank, world, port, mode, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from continuous_softmax_attention_gb300.dist import (cache_shard, context_ranges,
                                                             decode_context_parallel)
        from continuous_softmax_attention_gb300.inputs import make_decode_inputs

        x = make_decode_inputs(3, 2, 60, 8, seed=9, len_lo=1)
        T = x["k"].shape[2]
        lo, hi = context_ranges(T, world)[rank]
        ks, vs = cache_shard(x["k"], x["v"], lo, hi)

        def partial(qq, k_shard, v_shard, TT, a, b, k0, v0, *, seqlens, mode, scale):
            # the oracle stands in for csa_decode_range (it reads the whole cache)
            assert (a, b) == (lo, hi) and k_shard.shape[2] == ks.shape[2] and TT == T
            o, lse = oracle.decode_range(qq, x["k"], x["v"], seqlens, a, b, k0, v0, scale=scale,
                                         mode=mode)
            return torch.from_numpy(o), torch.from_numpy(lse)

        o, lse = decode_context_parallel(x["q"], ks, vs, T, x["k0"], x["v0"],
                                         seqlens=x["seqlens"], mode=mode, scale=0.7, fn=partial,
                                         merge_fn=_merge_np)
        q.put((rank, o.numpy(), lse.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,mode", [(2, 0), (3, 1), (3, 2), (4, 2)])
def test_decode_context_parallel_gloo(world, mode):
    """The cache split along time over 2 to 4 ranks: each rank's partial over
    its positions, one all-gather, the lse-weighted merge; every rank ends
    with the whole decode step."""
    from continuous_softmax_attention_gb300.inputs import make_decode_inputs

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, world, port, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = make_decode_inputs(3, 2, 60, 8, seed=9, len_lo=1)
    ro, rl = _oracle_decode(x["q"].float(), x["k"].float(), x["v"].float(), x["k0"].float(),
                            x["v0"].float(), x["seqlens"], mode, 0.7)
    for _, o, lse in got:
        assert np.abs(o - ro.numpy()).max() < 1e-9
        assert np.abs(lse - rl.numpy()).max() < 1e-9


def test_context_ranges_and_shards():
    from continuous_softmax_attention_gb300.dist import cache_shard, context_ranges

    for T in (3, 7, 60, 125, 126, 127, 8192):
        for world in range(1, min(8, (T + 1) // 2) + 1):
            rs = context_ranges(T, world)
            assert rs[0][0] == 0 and rs[-1][1] == T + 1 and len(rs) == world
            assert all(a < b for a, b in rs)
            assert all(b1 == a2 for (_, b1), (a2, _) in zip(rs, rs[1:]))
            assert all(a != 1 for a, _ in rs)  # never right after the sink
    with pytest.raises(ValueError):
        context_ranges(2, 2)
    k = torch.arange(2 * 1 * 10 * 4, dtype=torch.float32).reshape(2, 1, 10, 4)
    for lo, hi in ((0, 4), (4, 8), (8, 11), (2, 3)):
        ks, vs = cache_shard(k, k, lo, hi)
        r0, r1 = max(lo - 2, 0), min(hi, 10)
        assert torch.equal(ks, k[:, :, r0:r1]) and ks.is_contiguous()
        # the rows of the range's positions and of its two neighbours
        need = {p - 1 for p in range(max(lo - 1, 1), min(hi + 1, 11))}
        assert need == set(range(r0, r1))
