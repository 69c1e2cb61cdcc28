"""csa_decode_noalloc: the decode step with the library's fixed scratch
array instead of a caller workspace.  Called through the C ABI (ctypes) and
compared bit for bit with csa_decode on the same inputs, twice in a row, so
that a second call on the already-used scratch is covered too."""
import ctypes

import pytest
import torch

from continuous_softmax_attention_gb300 import _lib as L
from continuous_softmax_attention_gb300 import decode, decode_workspace_bytes
from continuous_softmax_attention_gb300.inputs import make_decode_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20  # CSA_DECODE_NOALLOC_SCRATCH_BYTES in include/csa.h


def _noalloc(lib, g, out, lse, B, H, T, d, scale, mode):
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.csa_decode_noalloc(ptr(g["q"]), ptr(g["k"]), ptr(g["v"]), ptr(g["k0"]),
                                  ptr(g["v0"]), ptr(g["seqlens"]), ptr(out), ptr(lse), B, H, T, d,
                                  ctypes.c_float(scale), mode,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _bind(lib):
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.csa_decode_noalloc.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, ctypes.c_float, i, p]
    lib.csa_decode_noalloc.restype = i
    return lib


@pytest.mark.parametrize("d,mode", [(128, 0), (64, 2), (256, 1)])
def test_noalloc_equals_workspace_entry_point_twice(d, mode):
    lib = _bind(L.load())
    B, H, T = 5, 3, 1100
    x = make_decode_inputs(B, H, T, d, seed=90 + d, len_lo=1)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / d ** 0.5
    for call in range(2):
        ref_o, ref_l = decode(g["q"], g["k"], g["v"], g["k0"], g["v0"], seqlens=g["seqlens"],
                              mode=mode, scale=scale)
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        free_before = torch.cuda.mem_get_info()[0]
        alloc_before = torch.cuda.memory_allocated()
        rc = _noalloc(lib, g, out, lse, B, H, T, d, scale, mode)
        torch.cuda.synchronize()
        assert rc == 0, L.status_string(rc)
        # nothing taken from torch's caching allocator, on any call
        assert torch.cuda.memory_allocated() == alloc_before
        if call == 1:  # scratch set up by now: the call must not take device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(out, ref_o), f"call {call}: outputs differ"
        assert torch.equal(lse, ref_l), f"call {call}: lse differs"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _bind(L.load())
    B, H, d = 64, 64, 128
    T = 16384
    assert decode_workspace_bytes(B, H, T, d) > SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before any launch
    rc = lib.csa_decode_noalloc(fake, fake, fake, None, None, None, fake, None, B, H, T, d,
                                ctypes.c_float(0.1), 0, None)
    assert rc == L.CSA_ERR_UNSUPPORTED
    # a size within the scratch still runs afterwards
    x = make_decode_inputs(1, 1, 300, d, seed=3)
    g = {k: t.cuda() for k, t in x.items()}
    out = torch.empty(1, 1, d, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, g, out, None, 1, 1, 300, d, 0.1, 0) == 0
    torch.cuda.synchronize()


def test_noalloc_at_and_just_past_its_capacity():
    """The largest size that fits the scratch (B*H*S*(d+2)*4 bytes, S the
    chunks of a row: 2^26 is not reachable, 264 bytes short is) runs and
    matches csa_decode bit for bit; one more head does not fit and is
    rejected before any launch."""
    lib = _bind(L.load())
    d, T, B = 128, 1, 1
    H_fit = SCRATCH_BYTES // ((d + 2) * 4)  # one chunk per row at T = 1
    assert decode_workspace_bytes(B, H_fit, T, d) <= SCRATCH_BYTES
    assert decode_workspace_bytes(B, H_fit + 1, T, d) > SCRATCH_BYTES
    x = make_decode_inputs(B, H_fit, T, d, seed=7, len_lo=1)
    g = {k: t.cuda() for k, t in x.items()}
    ref_o, ref_l = decode(g["q"], g["k"], g["v"], seqlens=g["seqlens"], scale=0.1)
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    rc = _noalloc(lib, g, out, lse, B, H_fit, T, d, 0.1, 0)
    torch.cuda.synchronize()
    assert rc == 0, L.status_string(rc)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before any launch
    rc = lib.csa_decode_noalloc(fake, fake, fake, None, None, None, fake, None, B, H_fit + 1, T, d,
                                ctypes.c_float(0.1), 0, None)
    assert rc == L.CSA_ERR_UNSUPPORTED


def test_noalloc_checks_arguments_before_its_capacity():
    """An oversized call with a bad argument gets csa_decode's error for that
    argument, not the capacity's."""
    lib = _bind(L.load())
    fake = ctypes.c_void_p(1 << 20)
    B, H, T, d = 64, 64, 16384, 128
    assert decode_workspace_bytes(B, H, T, d) > SCRATCH_BYTES
    call = lambda q=fake, mode=0, scale=0.1: lib.csa_decode_noalloc(
        q, fake, fake, None, None, None, fake, None, B, H, T, d, ctypes.c_float(scale), mode, None)
    assert call() == L.CSA_ERR_UNSUPPORTED
    assert call(q=None) == L.CSA_ERR_INVALID_ARG
    assert call(mode=7) == L.CSA_ERR_INVALID_ARG
    assert call(mode=2) == L.CSA_ERR_INVALID_ARG  # given sink without k0, v0
    assert call(scale=float("inf")) == L.CSA_ERR_INVALID_ARG
    assert call(q=ctypes.c_void_p((1 << 20) + 2)) == L.CSA_ERR_ALIGNMENT


def test_noalloc_argument_errors_match_decode():
    lib = _bind(L.load())
    fake = ctypes.c_void_p(1 << 20)
    call = lambda **kw: lib.csa_decode_noalloc(
        kw.get("q", fake), fake, fake, None, None, None, fake, None, kw.get("B", 1), 1,
        kw.get("T", 10), kw.get("d", 64), ctypes.c_float(0.1), kw.get("mode", 0), None)
    assert call(d=96) == L.CSA_ERR_UNSUPPORTED
    assert call(T=0) == L.CSA_ERR_INVALID_ARG
    assert call(B=0) == L.CSA_OK
    assert call(q=None) == L.CSA_ERR_INVALID_ARG
    assert call(mode=2) == L.CSA_ERR_INVALID_ARG
