"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library must load, export every function include/csa.h declares, and
reject bad arguments with the documented codes before touching the device."""
import ctypes
import os
import subprocess

import pytest

from continuous_softmax_attention_gb300 import _lib as L

FAKE = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
NULL = None


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from continuous_softmax_attention_gb300 import build

        build.build()
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = L.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True)
    exported = {line.split()[-1] for line in out.stdout.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_status_strings(lib):
    assert lib.csa_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.status_string(code) not in ("", "unknown status")
    assert L.status_string(123) == "unknown status"


def fwd(lib, *, q=FAKE, k=FAKE, v=FAKE, k0=NULL, v0=NULL, out=FAKE, lse=NULL, B=1, H=1, T=8, d=64,
        scale=0.125, mode=0):
    return lib.csa_forward(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, None)


def test_argument_validation(lib):
    assert fwd(lib, q=NULL) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, out=NULL) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, B=-1) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, d=0) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, mode=3) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, mode=2) == L.CSA_ERR_INVALID_ARG  # given sink without k0/v0
    assert fwd(lib, scale=float("nan")) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("inf")) == L.CSA_ERR_INVALID_ARG
    assert fwd(lib, d=300) == L.CSA_ERR_UNSUPPORTED
    assert fwd(lib, q=ctypes.c_void_p(4098)) == L.CSA_ERR_ALIGNMENT
    assert fwd(lib, out=ctypes.c_void_p(4104)) == L.CSA_ERR_ALIGNMENT


def test_empty_problems_are_ok(lib):
    # nothing to compute: success without any pointer or device
    assert fwd(lib, q=NULL, k=NULL, v=NULL, out=NULL, B=0) == L.CSA_OK
    assert fwd(lib, q=NULL, k=NULL, v=NULL, out=NULL, T=0) == L.CSA_OK
    assert lib.csa_std_forward(NULL, NULL, NULL, NULL, NULL, 2, 0, 5, 64, 0.1, None) == L.CSA_OK
    assert lib.csa_logphi2_eval(NULL, NULL, 0, None) == L.CSA_OK
    assert lib.csa_logphi2_eval(NULL, NULL, -1, None) == L.CSA_ERR_INVALID_ARG


def test_std_and_f32_validation(lib):
    assert lib.csa_std_forward(FAKE, FAKE, NULL, FAKE, NULL, 1, 1, 4, 64, 0.1, None) == L.CSA_ERR_INVALID_ARG
    assert lib.csa_forward_f32(FAKE, FAKE, FAKE, NULL, NULL, FAKE, NULL, 1, 1, 4, 257, 0.1, 0, None) == L.CSA_ERR_UNSUPPORTED
    assert lib.csa_forward_f32(ctypes.c_void_p(4097), FAKE, FAKE, NULL, NULL, FAKE, NULL, 1, 1, 4, 16, 0.1, 0, None) == L.CSA_ERR_ALIGNMENT
    assert lib.csa_selftest_wait_timeout(0, None) == L.CSA_ERR_INVALID_ARG
    assert lib.csa_selftest_wait_timeout(2000000, None) == L.CSA_ERR_INVALID_ARG
    # the planted-delay forward: delay above 10^6 ns or a half other than 0, 1
    dly = lambda **kw: lib.csa_selftest_forward_delay(
        FAKE, FAKE, FAKE, NULL, NULL, FAKE, NULL, 1, 1, 4, kw.get("d", 64), 0.1, 0,
        kw.get("ns", 1000), kw.get("half", 0), None)
    assert dly(ns=1000001) == L.CSA_ERR_INVALID_ARG
    assert dly(half=2) == L.CSA_ERR_INVALID_ARG
    assert dly(half=-1) == L.CSA_ERR_INVALID_ARG
    assert dly(d=96) == L.CSA_ERR_UNSUPPORTED


def test_no_device_is_reported(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments: the call reaches the device check and stops there
    assert fwd(lib) == L.CSA_ERR_NO_DEVICE
    assert lib.csa_device_status() == L.CSA_ERR_NO_DEVICE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        L.load()


def dec(lib, *, q=FAKE, k=FAKE, v=FAKE, k0=NULL, v0=NULL, seqlens=NULL, out=FAKE, lse=NULL,
        ws=FAKE, ws_bytes=1 << 30, B=2, H=2, T=300, d=128, scale=0.1, mode=0):
    return lib.csa_decode(q, k, v, k0, v0, seqlens, out, lse, ws, ws_bytes, B, H, T, d, scale,
                          mode, None)


def test_decode_workspace_bytes(lib):
    # one chunk of C positions (16384/d - 2; 110 at d = 256) per CTA over positions 0..T, each
    # leaving d partial outputs plus (max, sum): B*H*(T//C + 1)*(d + 2) floats
    for d, C in ((64, 254), (128, 126), (256, 110)):
        for T in (1, C - 1, C, C + 1, 8192):
            assert lib.csa_decode_workspace_bytes(3, 5, T, d) == 15 * (T // C + 1) * (d + 2) * 4
    assert lib.csa_decode_workspace_bytes(0, 5, 10, 64) == 0
    assert lib.csa_decode_workspace_bytes(1, 1, 10, 96) == -1
    assert lib.csa_decode_workspace_bytes(1, -1, 10, 64) == -1
    # positions 0..T counted in 64 bits: no overflow at the largest T
    imax = 2 ** 31 - 1
    assert lib.csa_decode_workspace_bytes(1, 1, imax, 128) == ((imax + 1 + 125) // 126) * 130 * 4
    assert lib.csa_decode_workspace_bytes(imax, imax, imax, 256) == -1  # beyond 2^62 bytes


def test_decode_validation(lib):
    need = lib.csa_decode_workspace_bytes(2, 2, 300, 128)
    assert dec(lib, q=NULL) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, ws=NULL) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, ws_bytes=need - 1) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, mode=2) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, mode=-1) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, scale=float("nan")) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, T=0) == L.CSA_ERR_INVALID_ARG  # a query needs its own key
    assert dec(lib, B=1, H=1, T=2 ** 31 - 1) == L.CSA_ERR_UNSUPPORTED  # positions 0..T
    assert dec(lib, d=96) == L.CSA_ERR_UNSUPPORTED
    assert dec(lib, d=0) == L.CSA_ERR_INVALID_ARG
    assert dec(lib, k=ctypes.c_void_p(4104)) == L.CSA_ERR_ALIGNMENT
    assert dec(lib, ws=ctypes.c_void_p(4100)) == L.CSA_ERR_ALIGNMENT
    assert dec(lib, mode=2, k0=ctypes.c_void_p(4098), v0=FAKE) == L.CSA_ERR_ALIGNMENT
    # empty batch: nothing to do, no pointer needed
    assert dec(lib, q=NULL, k=NULL, v=NULL, out=NULL, ws=NULL, B=0) == L.CSA_OK
    import torch

    if not torch.cuda.is_available():
        assert dec(lib, ws_bytes=need) == L.CSA_ERR_NO_DEVICE


def dec_range(lib, *, q=FAKE, k=FAKE, v=FAKE, k0=NULL, v0=NULL, seqlens=NULL, out=FAKE, lse=FAKE,
              ws=FAKE, ws_bytes=1 << 30, B=2, H=2, T=300, d=128, scale=0.1, mode=0, lo=0, hi=150):
    return lib.csa_decode_range(q, k, v, k0, v0, seqlens, out, lse, ws, ws_bytes, B, H, T, d,
                                scale, mode, lo, hi, None)


def test_decode_range_workspace_bytes(lib):
    # the range's chunks of C positions: ceil((hi - lo) / C) per (b, h)
    for d, C in ((64, 254), (128, 126), (256, 110)):
        for lo, hi in ((0, 1), (0, C), (0, C + 1), (2, 2 + C), (500, 8193)):
            n = -(-(hi - lo) // C)
            assert lib.csa_decode_range_workspace_bytes(3, 5, lo, hi, d) == 15 * n * (d + 2) * 4
        # a range over all positions needs what csa_decode needs
        assert (lib.csa_decode_range_workspace_bytes(2, 3, 0, 8193, d)
                == lib.csa_decode_workspace_bytes(2, 3, 8192, d))
    assert lib.csa_decode_range_workspace_bytes(1, 1, 5, 4, 64) == -1
    assert lib.csa_decode_range_workspace_bytes(1, 1, -1, 4, 64) == -1
    assert lib.csa_decode_range_workspace_bytes(1, 1, 0, 4, 96) == -1


def test_decode_range_validation(lib):
    assert dec_range(lib, lo=1, hi=100) == L.CSA_ERR_INVALID_ARG  # right after the sink
    assert dec_range(lib, lo=-1) == L.CSA_ERR_INVALID_ARG
    assert dec_range(lib, lo=100, hi=100) == L.CSA_ERR_INVALID_ARG
    assert dec_range(lib, lo=0, hi=302) == L.CSA_ERR_INVALID_ARG  # positions 0..T only
    assert dec_range(lib, lse=NULL) == L.CSA_ERR_INVALID_ARG  # the merge needs lse
    assert dec_range(lib, q=NULL) == L.CSA_ERR_INVALID_ARG
    assert dec_range(lib, ws_bytes=16) == L.CSA_ERR_INVALID_ARG
    assert dec_range(lib, mode=2) == L.CSA_ERR_INVALID_ARG
    assert dec_range(lib, d=96) == L.CSA_ERR_UNSUPPORTED
    assert dec_range(lib, out=ctypes.c_void_p(4104)) == L.CSA_ERR_ALIGNMENT
    assert dec_range(lib, k=NULL, v=NULL, q=NULL, out=NULL, lse=NULL, ws=NULL, B=0) == L.CSA_OK
    m = lambda **kw: lib.csa_decode_merge_ranges(kw.get("o", FAKE), kw.get("l", FAKE),
                                                 kw.get("R", 2), 2, 2, kw.get("d", 128),
                                                 kw.get("out", FAKE), NULL, None)
    assert m(R=0) == L.CSA_ERR_INVALID_ARG
    assert m(d=300) == L.CSA_ERR_INVALID_ARG
    assert m(o=NULL) == L.CSA_ERR_INVALID_ARG
    assert m(out=ctypes.c_void_p(4097)) == L.CSA_ERR_ALIGNMENT
    import torch

    if not torch.cuda.is_available():
        assert dec_range(lib) == L.CSA_ERR_NO_DEVICE
        assert m() == L.CSA_ERR_NO_DEVICE


def bwd(lib, *, q=FAKE, k=FAKE, v=FAKE, k0=NULL, v0=NULL, out=FAKE, lse=FAKE, dout=FAKE,
        dq=FAKE, dk=FAKE, dv=FAKE, dk0=NULL, dv0=NULL, ws=FAKE, ws_bytes=1 << 30, B=1, H=2, T=8,
        d=64, scale=0.1, mode=0):
    return lib.csa_backward(q, k, v, k0, v0, out, lse, dout, dq, dk, dv, dk0, dv0, ws, ws_bytes,
                            B, H, T, d, scale, mode, None)


def test_backward_validation(lib):
    need = lib.csa_backward_workspace_bytes(1, 2, 8, 64)
    assert need == 2 * 1 * 2 * 8 * 64 * 4  # fp32 dk, dv accumulators
    assert lib.csa_backward_workspace_bytes(1, 1, 1, 257) == -1
    assert bwd(lib, lse=NULL) == L.CSA_ERR_INVALID_ARG
    assert bwd(lib, dout=NULL) == L.CSA_ERR_INVALID_ARG
    assert bwd(lib, ws=NULL) == L.CSA_ERR_INVALID_ARG
    assert bwd(lib, ws_bytes=need - 1) == L.CSA_ERR_INVALID_ARG
    assert bwd(lib, mode=2, k0=FAKE, v0=FAKE) == L.CSA_ERR_INVALID_ARG  # no dk0/dv0
    assert bwd(lib, d=300) == L.CSA_ERR_UNSUPPORTED
    assert bwd(lib, dq=ctypes.c_void_p(4097)) == L.CSA_ERR_ALIGNMENT
    assert bwd(lib, q=NULL, k=NULL, v=NULL, out=NULL, lse=NULL, dout=NULL, dq=NULL, dk=NULL,
               dv=NULL, ws=NULL, T=0) == L.CSA_OK
    import torch

    if not torch.cuda.is_available():
        assert bwd(lib, ws_bytes=need) == L.CSA_ERR_NO_DEVICE


def test_forward_host_validation(lib):
    need = lib.csa_forward_host_workspace_bytes(1, 4, 16, 64)
    # q, k, v, out bf16 and lse fp32, each rounded up to 256 bytes
    assert need == 4 * (4 * 16 * 64 * 2) + 256
    call = lambda **kw: lib.csa_forward_host(
        kw.get("q", FAKE), FAKE, FAKE, None, None, FAKE, None, kw.get("ws", ctypes.c_void_p(1 << 20)),
        kw.get("ws_bytes", need), 1, 4, 16, 64, ctypes.c_float(0.1), 0, kw.get("hpc", 2), None,
        None, None)
    lib.csa_forward_host.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_longlong] + [ctypes.c_int] * 4 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 3
    assert call(hpc=3) == L.CSA_ERR_INVALID_ARG  # does not divide H
    assert call(hpc=0) == L.CSA_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == L.CSA_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == L.CSA_ERR_ALIGNMENT
    assert call(q=NULL) == L.CSA_ERR_INVALID_ARG
    ex = lambda flags: lib.csa_forward_host_ex(
        FAKE, FAKE, FAKE, None, None, FAKE, None, ctypes.c_void_p(1 << 20), need, 1, 4, 16, 64,
        ctypes.c_float(0.1), 0, 2, flags, None, None, None)
    assert ex(2) == L.CSA_ERR_INVALID_ARG  # unknown flag bit
    assert ex(0x80000000) == L.CSA_ERR_INVALID_ARG
    import torch

    if not torch.cuda.is_available():
        assert call() == L.CSA_ERR_NO_DEVICE
        assert ex(0) == L.CSA_ERR_NO_DEVICE
        assert ex(L.CSA_HOST_NO_ENTRY_WAIT) == L.CSA_ERR_NO_DEVICE
