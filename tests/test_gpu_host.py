"""csa_forward_host: the forward pass from pinned host buffers with the
copies overlapped by chunks of heads.  Each (b, h) problem runs the same
kernel code as csa_forward, so the results must match it bit for bit."""
import pytest
import torch

from continuous_softmax_attention_gb300 import forward, forward_host, forward_host_workspace_bytes
from continuous_softmax_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def pinned(t):
    return t.contiguous().pin_memory()


def host_run(x, mode, hpc, streams=True, want_lse=True):
    B, H, T, d = x["q"].shape
    ws = torch.empty(forward_host_workspace_bytes(B, H, T, d), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, H, T, d, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty(B, H, T).pin_memory() if want_lse else None
    s1 = torch.cuda.Stream() if streams else None
    s2 = torch.cuda.Stream() if streams else None
    forward_host(pinned(x["q"]), pinned(x["k"]), pinned(x["v"]), out, lse, x["k0"].cuda(),
                 x["v0"].cuda(), mode=mode, workspace=ws, heads_per_chunk=hpc, stream_h2d=s1,
                 stream_d2h=s2)
    torch.cuda.current_stream().synchronize()
    return out, lse


@pytest.mark.parametrize("d,mode,hpc", [(128, 0, 1), (128, 2, 2), (64, 1, 4), (96, 2, 2)])
def test_host_path_matches_device_path(d, mode, hpc):
    x = make_inputs(2, 4, 300, d, "bf16", seed=400 + d + mode)
    o, lse = host_run(x, mode, hpc)
    g = {k: t.cuda() for k, t in x.items()}
    ro, rl = forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu()) and torch.equal(lse, rl.cpu())


def test_host_path_single_stream_and_no_lse():
    x = make_inputs(1, 4, 200, 128, "bf16", seed=410)
    o, _ = host_run(x, 0, 4, streams=False, want_lse=False)
    g = {k: t.cuda() for k, t in x.items()}
    ro, _ = forward(g["q"], g["k"], g["v"])
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu())


def test_host_path_back_to_back_calls():
    """A second call with new inputs queued right behind the first must not
    disturb it (the copies wait for the compute stream's earlier work)."""
    B, H, T, d = 1, 8, 1024, 128
    xa = make_inputs(B, H, T, d, "bf16", seed=420)
    xb = make_inputs(B, H, T, d, "bf16", seed=421)
    ws = torch.empty(forward_host_workspace_bytes(B, H, T, d), dtype=torch.uint8, device="cuda")
    outs = [torch.empty(B, H, T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for x, o in zip((xa, xb), outs):
        forward_host(pinned(x["q"]), pinned(x["k"]), pinned(x["v"]), o, None, workspace=ws,
                     heads_per_chunk=2, stream_h2d=s1, stream_d2h=s2)
    torch.cuda.current_stream().synchronize()
    for x, o in zip((xa, xb), outs):
        g = {k: t.cuda() for k, t in x.items()}
        ro, _ = forward(g["q"], g["k"], g["v"])
        torch.cuda.synchronize()
        assert torch.equal(o, ro.cpu())


def test_host_path_rejects_bad_chunks():
    x = make_inputs(1, 4, 16, 64, "bf16", seed=430)
    ws = torch.empty(forward_host_workspace_bytes(1, 4, 16, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty(1, 4, 16, 64, dtype=torch.bfloat16)
    from continuous_softmax_attention_gb300 import CsaError

    for hpc in (0, 3, 5):
        with pytest.raises(CsaError):
            forward_host(x["q"], x["k"], x["v"], out, workspace=ws, heads_per_chunk=hpc)


def test_back_to_back_calls_overlapped_across_calls():
    """Five calls in a row, each on different inputs, through the two-workspace
    pipeline (copies in without the entry wait): every result must still equal
    the device path bit for bit, so no call overwrote a workspace or an output
    another call was still using."""
    from continuous_softmax_attention_gb300 import HostForwardPipeline

    B, H, T, d = 1, 8, 640, 128
    pipe = HostForwardPipeline(B, H, T, d, "cuda", heads_per_chunk=2)
    runs = []
    for i in range(5):
        x = make_inputs(B, H, T, d, "bf16", seed=900 + i)
        out = torch.empty(B, H, T, d, dtype=torch.bfloat16).pin_memory()
        lse = torch.empty(B, H, T).pin_memory()
        # the pinned inputs stay referenced until the copies have run
        hq, hk, hv = pinned(x["q"]), pinned(x["k"]), pinned(x["v"])
        pipe(hq, hk, hv, out, lse, mode=0)
        runs.append((x, out, lse, (hq, hk, hv)))
    torch.cuda.current_stream().synchronize()
    for x, out, lse, _ in runs:
        g = {k: t.cuda() for k, t in x.items()}
        ro, rl = forward(g["q"], g["k"], g["v"], mode=0)
        torch.cuda.synchronize()
        assert torch.equal(out, ro.cpu()) and torch.equal(lse, rl.cpu())
