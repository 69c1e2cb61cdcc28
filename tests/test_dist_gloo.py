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


@pytest.mark.parametrize("B,H,mode", [(2, 3, 2), (1, 5, 0), (3, 1, 1)])
def test_two_gloo_ranks_match_single_process(B, H, mode):
    import oracle
    from continuous_softmax_attention_gb300.inputs import make_inputs

    T, d, world = 40, 8, 2
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
    assert t == 11.0


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
