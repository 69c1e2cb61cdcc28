"""GPU parity of the CUDA kernels against the CPU oracle at sizes the oracle
finishes in seconds, spanning several tiles and ragged tails, plus the
invariants that must hold bit for bit (determinism, causality, canaries).

Calls go through the C ABI (ctypes binding).  Every input comes from the
seeded generator; every expected value from the oracle."""
import math

import numpy as np
import pytest
import torch

import continuous_softmax_attention_gb300 as csa
import oracle
from oracle import quadrature
from continuous_softmax_attention_gb300.inputs import make_inputs
from gpu_util import assert_close, np64, to_dev

pytestmark = pytest.mark.gpu

MODES = [csa.ZERO, csa.COPY_FIRST, csa.GIVEN]


def run_csa(x, mode, scale, dev_x=None):
    g = dev_x or to_dev(x)
    o, lse = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale)
    torch.cuda.synchronize()
    assert csa.device_status() == 0
    return o, lse


def oracle_csa(x, mode, scale):
    return oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=scale, mode=mode)


# ------------------------------------------------------------------ fp32 (CUDA cores)
def test_tiny_workload_f32_against_oracle_and_quadrature():
    """B=1, H=1, T=64, d=16, fp32, scale 1/4, zero sink; also against eq. (2)
    integrated numerically."""
    x = make_inputs(1, 1, 64, 16, "f32", seed=0)
    o, lse = run_csa(x, csa.ZERO, 0.25)
    ro, rl = oracle_csa(x, csa.ZERO, 0.25)
    assert_close(o, lse, ro, rl, "f32", "tiny vs oracle")
    qo, ql = quadrature.forward(x["q"].numpy(), x["k"].numpy(), x["v"].numpy(), scale=0.25)
    assert_close(o, lse, qo, ql, "f32", "tiny vs quadrature")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,d,scale", [(1, 16, 0.5), (37, 8, 1.0), (130, 64, 0.125), (200, 100, 0.3),
                                       (70, 256, 0.05), (90, 32, 3.0)])
def test_f32_kernel(mode, T, d, scale):
    x = make_inputs(2, 3, T, d, "f32", seed=T + d)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "f32", f"f32 T={T} d={d}")


@pytest.mark.parametrize("T,d", [(1, 16), (50, 64), (130, 128), (77, 200)])
def test_std_f32_kernel(T, d):
    x = make_inputs(2, 2, T, d, "f32", seed=5 + T)
    g = to_dev(x)
    o, lse = csa.std_forward(g["q"], g["k"], g["v"], scale=0.2)
    torch.cuda.synchronize()
    ro, rl = oracle.std_forward(x["q"], x["k"], x["v"], scale=0.2)
    assert_close(o, lse, ro, rl, "f32", "std f32")


# ------------------------------------------------------------------ bf16 tensor cores
# Lengths around every tile edge of the tensor-core kernels: 128-row query
# tiles in 256-row pairs, key tiles every 110 keys (d = 128) or 126 (d = 64).
TC_SHAPES = [(128, 1), (128, 2), (128, 3), (128, 108), (128, 109), (128, 110), (128, 111),
             (128, 126), (128, 127), (128, 128), (128, 129), (128, 219), (128, 220), (128, 221),
             (128, 254), (128, 255), (128, 256), (128, 257), (128, 383), (128, 385), (128, 700),
             (64, 1), (64, 5), (64, 124), (64, 125), (64, 126), (64, 127), (64, 128), (64, 251),
             (64, 252), (64, 255), (64, 258), (64, 513)]


@pytest.mark.parametrize("d,T", TC_SHAPES)
@pytest.mark.parametrize("mode", MODES)
def test_tc_kernel_shapes(d, T, mode):
    x = make_inputs(2, 3, T, d, "bf16", seed=1000 + 7 * T + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "bf16", f"tc d={d} T={T} mode={mode}")


@pytest.mark.parametrize("d,T", [(128, 1), (128, 127), (128, 128), (128, 129), (128, 300),
                                 (128, 513), (64, 2), (64, 129), (64, 400)])
def test_tc_std_kernel(d, T):
    x = make_inputs(2, 2, T, d, "bf16", seed=2000 + T + d)
    g = to_dev(x)
    scale = 1.0 / math.sqrt(d)
    o, lse = csa.std_forward(g["q"], g["k"], g["v"], scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.std_forward(x["q"], x["k"], x["v"], scale=scale)
    assert_close(o, lse, ro, rl, "bf16", f"std tc d={d} T={T}")
    # and against torch's own fused attention on the same device
    ref = torch.nn.functional.scaled_dot_product_attention(g["q"], g["k"], g["v"], is_causal=True,
                                                           scale=scale)
    assert (o.float() - ref.float()).abs().max().item() < 2e-2


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0])
@pytest.mark.parametrize("mode", [csa.ZERO, csa.COPY_FIRST])
def test_stress_workload(scale, mode):
    """B=2, H=4, T=512, d=64, bf16; scale in {1/8, 1, 4} (logit steps up to
    about +-200 at 4) x {zero, copy-first} sink, full comparison."""
    x = make_inputs(2, 4, 512, 64, "bf16", seed=1)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "bf16", f"stress scale={scale} mode={mode}")


@pytest.mark.parametrize("scale", [0.125, 1.0, 4.0])
@pytest.mark.parametrize("mode", MODES)
def test_stress_scales_d128(scale, mode):
    """The stress workload's scales at d = 128 (112-key tiles, several
    running-max raises per row at scale 4), B=2, H=4, T=512, every sink
    mode, full comparison."""
    x = make_inputs(2, 4, 512, 128, "bf16", seed=2)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "bf16", f"d=128 stress scale={scale} mode={mode}")


@pytest.mark.parametrize("d", [64, 128])
def test_tc_matches_cuda_core_log_domain_path(d):
    """The tensor-core kernel (interval weights R, L) against the CUDA-core
    kernel (log-domain b with log phi2 and logaddexp) on identical values."""
    x = make_inputs(1, 4, 600, d, "bf16", seed=77 + d)
    g = to_dev(x)
    scale = 1.0 / math.sqrt(d)
    o_tc, l_tc = csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=csa.GIVEN, scale=scale)
    f = {k: v.float() for k, v in g.items()}
    o_f, l_f = csa.forward(f["q"], f["k"], f["v"], f["k0"], f["v0"], mode=csa.GIVEN, scale=scale)
    torch.cuda.synchronize()
    assert_close(o_tc, l_tc, np64(o_f), np64(l_f), "bf16", "tc vs cuda-core")


def test_bf16_cuda_core_kernel_other_head_dims():
    """bf16 with d outside {64, 128} runs on the CUDA-core kernel."""
    for d in (32, 96, 160):
        x = make_inputs(1, 2, 150, d, "bf16", seed=d)
        for mode in MODES:
            o, lse = run_csa(x, mode, 0.2)
            ro, rl = oracle_csa(x, mode, 0.2)
            assert_close(o, lse, ro, rl, "bf16", f"simt bf16 d={d}")


def test_equal_logits_trapezoid():
    """scale = 0: the trapezoid rule (oracle) exactly reproduced within bf16."""
    x = make_inputs(1, 2, 300, 128, "bf16", seed=3)
    for mode in MODES:
        o, lse = run_csa(x, mode, 0.0)
        ro, rl = oracle_csa(x, mode, 0.0)
        assert_close(o, lse, ro, rl, "bf16", "scale 0")
        t = np.arange(1, 301, dtype=np.float64)
        assert np.abs(np64(lse) - np.log(t)[None, None]).max() < 1e-3


def test_constant_values_copy_first():
    x = make_inputs(1, 2, 400, 128, "bf16", seed=4)
    c = torch.linspace(-2, 2, 128).to(torch.bfloat16)
    x["v"] = c.expand_as(x["v"]).contiguous()
    o, _ = run_csa(x, csa.COPY_FIRST, 1.0 / math.sqrt(128))
    assert (o.float().cpu() - c.float()).abs().max().item() < 2e-2


def test_determinism():
    x = make_inputs(1, 4, 700, 128, "bf16", seed=5)
    g = to_dev(x)
    o1, l1 = run_csa(x, csa.GIVEN, 0.1, g)
    o2, l2 = run_csa(x, csa.GIVEN, 0.1, g)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("cut", [0, 107, 108, 109, 110, 125, 126, 127, 128, 217, 218, 219, 253, 254,
                                 255, 300])
def test_causality_no_halo_leak(cut):
    """Changing keys/values after position `cut` leaves rows <= cut bit-identical
    (the halo column must not see past the diagonal)."""
    x = make_inputs(1, 2, 512, 128, "bf16", seed=6)
    o1, l1 = run_csa(x, csa.ZERO, 0.1)
    y = dict(x)
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["k"][:, :, cut + 1:] = (y["k"][:, :, cut + 1:].float() * 3 + 1).to(torch.bfloat16)
    y["v"][:, :, cut + 1:] = (y["v"][:, :, cut + 1:].float() - 5).to(torch.bfloat16)
    o2, l2 = run_csa(y, csa.ZERO, 0.1)
    assert torch.equal(o1[:, :, :cut + 1], o2[:, :, :cut + 1])
    assert torch.equal(l1[:, :, :cut + 1], l2[:, :, :cut + 1])


@pytest.mark.parametrize("continuous", [True, False])
def test_output_canaries(continuous):
    """Nothing is written outside out[B,H,T,d] and lse[B,H,T]."""
    B, H, T, d = 1, 3, 333, 128
    x = make_inputs(B, H, T, d, "bf16", seed=8)
    g = to_dev(x)
    pad = 64
    n = B * H * T * d
    big = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[pad:pad + n].view(B, H, T, d)
    lbig = torch.full((B * H * T + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    lse = lbig[pad:pad + B * H * T].view(B, H, T)
    if continuous:
        csa.forward(g["q"], g["k"], g["v"], mode=csa.ZERO, out=out, lse=lse)
    else:
        csa.std_forward(g["q"], g["k"], g["v"], out=out, lse=lse)
    torch.cuda.synchronize()
    assert (big[:pad] == 7).all() and (big[pad + n:] == 7).all()
    assert (lbig[:pad] == 7).all() and (lbig[pad + B * H * T:] == 7).all()
    assert torch.isfinite(out.float()).all()


def test_no_lse_requested():
    x = make_inputs(1, 1, 200, 64, "bf16", seed=9)
    g = to_dev(x)
    o, lse = csa.forward(g["q"], g["k"], g["v"], want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    ro, _ = oracle_csa(x, csa.ZERO, 0.125)
    assert np.abs(np64(o) - ro).max() < 2e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [-0.1, -1.0])
@pytest.mark.parametrize("mode", MODES)
def test_negative_scale(d, scale, mode):
    """The pages put no sign on the logits (eq. (2)): a negative scale runs on
    the tensor cores like any other."""
    x = make_inputs(1, 3, 300, d, "bf16", seed=10 + d)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "bf16", f"scale={scale} mode={mode} d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_std_negative_scale(d):
    x = make_inputs(1, 2, 300, d, "bf16", seed=20 + d)
    g = to_dev(x)
    o, lse = csa.std_forward(g["q"], g["k"], g["v"], scale=-0.3)
    torch.cuda.synchronize()
    ro, rl = oracle.std_forward(x["q"], x["k"], x["v"], scale=-0.3)
    assert_close(o, lse, ro, rl, "bf16", f"std scale<0 d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", MODES)
def test_running_max_raised(d, mode):
    """Keys far into the sequence whose logits exceed every earlier one by
    hundreds (log2 units): the kernel holds the first key tile's max until a
    16-key chunk's weights would pass 2^64, then raises it and rescales what
    it has written.  The oracle is exact for any logits."""
    T = 700
    x = make_inputs(1, 2, T, d, "bf16", seed=30 + d)
    k = x["k"].float()
    for pos, f in ((300, 25.0), (301, 25.0), (450, 60.0), (640, 90.0)):
        k[:, :, pos] = k[:, :, pos] * f
    x["k"] = k.to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_csa(x, mode, scale)
    ro, rl = oracle_csa(x, mode, scale)
    assert_close(o, lse, ro, rl, "bf16", f"max raised d={d} mode={mode}")
