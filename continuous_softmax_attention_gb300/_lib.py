"""ctypes binding of libcsa.so (C ABI declared in include/csa.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and torch's current stream are passed to the
C entry point, and a non-zero status becomes a CsaError.  Every step of the
computation runs in the library's CUDA kernels; there is no other path.  If
the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "csa.h")

CSA_OK = 0
CSA_ERR_INVALID_ARG = -1
CSA_ERR_UNSUPPORTED = -2
CSA_ERR_ALIGNMENT = -3
CSA_ERR_CUDA = -4
CSA_ERR_TIMEOUT = -5
CSA_ERR_NO_DEVICE = -6


class CsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


_lib = None


def load():
    """Loads libcsa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m continuous_softmax_attention_gb300.build` (no other compute path exists)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i, f, u = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint
    fwd = [p, p, p, p, p, p, p, i, i, i, i, f, i, p]
    std = [p, p, p, p, p, i, i, i, i, f, p]
    bwd = [p, p, p, p, p, p, p, p, p, p, p, p, p, p, ctypes.c_longlong, i, i, i, i, f, i, p]
    for name, args in (("csa_forward", fwd), ("csa_forward_f32", fwd),
                       ("csa_forward_short_conv", fwd), ("csa_forward_short_conv_f32", fwd),
                       ("csa_forward_logdomain", fwd),
                       ("csa_std_forward", std), ("csa_std_forward_f32", std),
                       ("csa_forward_symmetric", std), ("csa_forward_symmetric_f32", std),
                       ("csa_logphi2_eval", [p, p, i, p]),
                       ("csa_segment_weights_eval", [p, p, p, p, i, p]),
                       ("csa_device_status", []),
                       ("csa_selftest_wait_timeout", [u, p]),
                       ("csa_selftest_forward_delay", [p, p, p, p, p, p, p, i, i, i, i, f, i, u,
                                                       i, p]),
                       ("csa_abi_version", []),
                       ("csa_decode", [p, p, p, p, p, p, p, p, p, ctypes.c_longlong, i, i, i, i,
                                       f, i, p]),
                       ("csa_decode_noalloc", [p, p, p, p, p, p, p, p, i, i, i, i, f, i, p]),
                       ("csa_decode_range", [p, p, p, p, p, p, p, p, p, ctypes.c_longlong, i, i,
                                             i, i, f, i, i, i, p]),
                       ("csa_decode_merge_ranges", [p, p, i, i, i, i, p, p, p]),
                       ("csa_backward", bwd), ("csa_backward_f32", bwd),
                       ("csa_forward_host", [p, p, p, p, p, p, p, p, ctypes.c_longlong, i, i, i,
                                             i, f, i, i, p, p, p]),
                       ("csa_forward_host_ex", [p, p, p, p, p, p, p, p, ctypes.c_longlong, i, i,
                                                i, i, f, i, i, u, p, p, p])):
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i
    for name in ("csa_decode_workspace_bytes", "csa_backward_workspace_bytes",
                 "csa_forward_host_workspace_bytes"):
        getattr(lib, name).argtypes = [i, i, i, i]
        getattr(lib, name).restype = ctypes.c_longlong
    lib.csa_decode_range_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.csa_decode_range_workspace_bytes.restype = ctypes.c_longlong
    lib.csa_status_string.argtypes = [i]
    lib.csa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().csa_status_string(int(code)).decode()
    except Exception:  # library missing: fall back to the number
        return f"status {code}"


def header_functions(path: str = HEADER):
    """Names of the functions declared in include/csa.h."""
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", src)))


def _check(code: int, where: str):
    if code != CSA_OK:
        raise CsaError(code, where)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensor(t, name, dtype, shape, device):
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def forward(q, k, v, k0=None, v0=None, *, mode: int = 0, scale=None, out=None, lse=None,
            stream=None, want_lse: bool = True, short_conv: bool = False,
            log_domain: bool = False):
    """Causal continuous softmax attention.  Returns (o, lse).

    q, k, v: CUDA tensors [B, H, T, d], all bf16 (tensor-core kernel for
    d in {64, 128}) or all fp32 (CUDA-core kernel).  k0, v0: [H, d], read
    in mode GIVEN (2).  mode: 0 zero sink, 1 copy of the first token,
    2 given.  scale defaults to 1/sqrt(d).  short_conv=True runs the
    first-order (eq. (13)) reading instead (csa_forward_short_conv);
    log_domain=True forms the same weights as z = a + b in the log domain
    (csa_forward_logdomain; bf16 only: the fp32 kernel already does)."""
    import torch

    B, H, T, d = q.shape
    dtype, dev = q.dtype, q.device
    for name, t in (("k", k), ("v", v)):
        _check_tensor(t, name, dtype, (B, H, T, d), dev)
    _check_tensor(q, "q", dtype, (B, H, T, d), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", dtype, (H, d), dev)
        _check_tensor(v0, "v0", dtype, (H, d), dev)
    else:
        k0 = v0 = None
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out", dtype, (B, H, T, d), dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, H, T), dev)
    lib = load()
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"unsupported dtype {dtype}")
    if short_conv and log_domain:
        raise ValueError("short_conv and log_domain are separate forms")
    if log_domain and dtype != torch.bfloat16:
        raise ValueError("log_domain is a bf16 form (csa_forward_f32 forms b in the log domain)")
    where = ("csa_forward_short_conv" if short_conv else
             "csa_forward_logdomain" if log_domain else "csa_forward") + (
        "" if dtype == torch.bfloat16 else "_f32")
    fn = getattr(lib, where)
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(out), _ptr(lse),
              B, H, T, d, float(scale), int(mode), _stream_handle(stream)), where)
    return out, lse


def forward_host_workspace_bytes(B: int, H: int, T: int, d: int) -> int:
    """Device workspace bytes csa_forward_host needs (host-side)."""
    n = int(load().csa_forward_host_workspace_bytes(int(B), int(H), int(T), int(d)))
    if n < 0:
        raise CsaError(CSA_ERR_UNSUPPORTED, "csa_forward_host_workspace_bytes")
    return n


CSA_HOST_NO_ENTRY_WAIT = 1


def forward_host(q, k, v, out, lse=None, k0=None, v0=None, *, mode: int = 0, scale=None,
                 workspace=None, heads_per_chunk: int = 4, stream=None, stream_h2d=None,
                 stream_d2h=None, no_entry_wait: bool = False):
    """csa_forward from host tensors, end to end, with the copies overlapped.

    q, k, v, out: CPU bf16 [B, H, T, d] (pinned for the overlap); lse: CPU
    float32 [B, H, T] or None; k0, v0: CUDA [H, d] in mode GIVEN.
    workspace: CUDA uint8 tensor of forward_host_workspace_bytes(...) bytes.
    The call is asynchronous: out and lse are ready once `stream` (torch's
    current stream by default) has reached this point.  no_entry_wait: the
    copies in do not wait for work already queued on `stream`
    (csa_forward_host_ex with CSA_HOST_NO_ENTRY_WAIT); the caller orders the
    calls that share a workspace."""
    import torch

    B, H, T, d = q.shape
    cpu = torch.device("cpu")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_tensor(t, name, torch.bfloat16, (B, H, T, d), cpu)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, H, T), cpu)
    if workspace is None or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    dev = workspace.device
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", torch.bfloat16, (H, d), dev)
        _check_tensor(v0, "v0", torch.bfloat16, (H, d), dev)
    else:
        k0 = v0 = None
    if scale is None:
        scale = 1.0 / d ** 0.5
    nbytes = workspace.numel() * workspace.element_size()
    cs = _stream_handle(stream)
    hs = _stream_handle(stream_h2d) if stream_h2d is not None else cs
    ds = _stream_handle(stream_d2h) if stream_d2h is not None else cs
    flags = CSA_HOST_NO_ENTRY_WAIT if no_entry_wait else 0
    _check(load().csa_forward_host_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(out),
                                      _ptr(lse), _ptr(workspace), nbytes, B, H, T, d,
                                      float(scale), int(mode), int(heads_per_chunk), flags, cs,
                                      hs, ds),
           "csa_forward_host_ex")
    return out, lse


class HostForwardPipeline:
    """Back-to-back forward_host calls that overlap across calls: two
    workspaces used alternately, each call's copies in (CSA_HOST_NO_ENTRY_WAIT)
    waiting only for the call before last, which used the same workspace, to
    have completed on `stream`.  So one call's copies in run while the previous
    call's kernels and copies out do.  Stream and event plumbing only."""

    def __init__(self, B: int, H: int, T: int, d: int, device, *, heads_per_chunk: int = 4,
                 stream=None):
        import torch

        n = forward_host_workspace_bytes(B, H, T, d)
        self.ws = [torch.empty(max(n, 16), dtype=torch.uint8, device=device) for _ in range(2)]
        self.done = [None, None]
        self.s_h2d = torch.cuda.Stream(device=device)
        self.s_d2h = torch.cuda.Stream(device=device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(device)
        self.heads_per_chunk = heads_per_chunk
        self.calls = 0

    def __call__(self, q, k, v, out, lse=None, k0=None, v0=None, *, mode: int = 0, scale=None):
        import torch

        w = self.calls & 1
        if self.done[w] is not None:
            self.s_h2d.wait_event(self.done[w])
        forward_host(q, k, v, out, lse, k0, v0, mode=mode, scale=scale, workspace=self.ws[w],
                     heads_per_chunk=self.heads_per_chunk, stream=self.stream,
                     stream_h2d=self.s_h2d, stream_d2h=self.s_d2h, no_entry_wait=True)
        ev = torch.cuda.Event()
        ev.record(self.stream)
        self.done[w] = ev
        self.calls += 1
        return out, lse


def std_forward(q, k, v, *, scale=None, out=None, lse=None, stream=None, want_lse: bool = True,
                _entry: str = "csa_std_forward"):
    """Standard causal softmax attention (b = 0, no sink).  Returns (o, lse)."""
    import torch

    B, H, T, d = q.shape
    dtype, dev = q.dtype, q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, name, dtype, (B, H, T, d), dev)
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out", dtype, (B, H, T, d), dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, H, T), dev)
    lib = load()
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"unsupported dtype {dtype}")
    where = _entry + ("" if dtype == torch.bfloat16 else "_f32")
    fn = getattr(lib, where)
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, T, d, float(scale),
              _stream_handle(stream)), where)
    return out, lse


def forward_symmetric(q, k, v, *, scale=None, out=None, lse=None, stream=None,
                      want_lse: bool = True):
    """Continuous attention over the symmetric interval [1/2, t + 1/2]
    (constant end half-cells, no sink).  Returns (o, lse)."""
    return std_forward(q, k, v, scale=scale, out=out, lse=lse, stream=stream, want_lse=want_lse,
                       _entry="csa_forward_symmetric")


def decode_workspace_bytes(B: int, H: int, T: int, d: int) -> int:
    """Bytes of workspace csa_decode needs (host-side, no device needed)."""
    n = int(load().csa_decode_workspace_bytes(int(B), int(H), int(T), int(d)))
    if n < 0:
        raise CsaError(CSA_ERR_UNSUPPORTED, "csa_decode_workspace_bytes")
    return n


def decode(q, k_cache, v_cache, k0=None, v0=None, *, seqlens=None, mode: int = 0, scale=None,
           out=None, lse=None, workspace=None, stream=None, want_lse: bool = True):
    """One decode step: the newest token of each sequence against its cache.

    q: bf16 CUDA [B, H, d]; k_cache, v_cache: bf16 [B, H, T, d]; seqlens: int32
    CUDA [B] with the used lengths n_b (None: all T).  k0, v0: [H, d] in mode
    GIVEN (2).  workspace: a uint8 CUDA tensor of at least
    decode_workspace_bytes(B, H, T, d) bytes (allocated when None).
    Returns (o [B, H, d], lse [B, H])."""
    import torch

    B, H, T, d = k_cache.shape
    dev = k_cache.device
    bf = torch.bfloat16
    _check_tensor(k_cache, "k_cache", bf, (B, H, T, d), dev)
    _check_tensor(v_cache, "v_cache", bf, (B, H, T, d), dev)
    _check_tensor(q, "q", bf, (B, H, d), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", bf, (H, d), dev)
        _check_tensor(v0, "v0", bf, (H, d), dev)
    else:
        k0 = v0 = None
    if seqlens is not None:
        _check_tensor(seqlens, "seqlens", torch.int32, (B,), dev)
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty((B, H, d), dtype=bf, device=dev)
    _check_tensor(out, "out", bf, (B, H, d), dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, H), dev)
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_bytes(B, H, T, d), 16), dtype=torch.uint8,
                                device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the cache's device")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().csa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k0), _ptr(v0),
                             _ptr(seqlens), _ptr(out), _ptr(lse), _ptr(workspace), nbytes, B, H,
                             T, d, float(scale), int(mode), _stream_handle(stream)), "csa_decode")
    return out, lse


def decode_range_workspace_bytes(B: int, H: int, pos_lo: int, pos_hi: int, d: int) -> int:
    """Bytes of workspace csa_decode_range needs (host-side, no device needed)."""
    n = int(load().csa_decode_range_workspace_bytes(int(B), int(H), int(pos_lo), int(pos_hi),
                                                    int(d)))
    if n < 0:
        raise CsaError(CSA_ERR_UNSUPPORTED, "csa_decode_range_workspace_bytes")
    return n


def shard_rows(T: int, pos_lo: int, pos_hi: int):
    """Cache rows [start, stop) a range's shard holds: its positions and one
    neighbour on each side (position i >= 1 is cache row i - 1)."""
    return max(pos_lo - 2, 0), min(pos_hi, T)


def decode_range(q, k_shard, v_shard, T: int, pos_lo: int, pos_hi: int, k0=None, v0=None, *,
                 seqlens=None, mode: int = 0, scale=None, out=None, lse=None, workspace=None,
                 stream=None):
    """The decode step over the positions [pos_lo, pos_hi) of each row only
    (csa_decode_range): one range of a cache split along its time axis.

    q: bf16 CUDA [B, H, d]; k_shard, v_shard: bf16 [B, H, rows, d] holding the
    cache rows shard_rows(T, pos_lo, pos_hi); T: the whole cache's capacity.
    Returns (o_r fp32 [B, H, d], lse_r fp32 [B, H]) for decode_merge_ranges."""
    import torch

    B, H, rows, d = k_shard.shape
    dev = k_shard.device
    bf = torch.bfloat16
    r0, r1 = shard_rows(T, pos_lo, pos_hi)
    if rows != r1 - r0:
        raise ValueError(f"the shard of positions [{pos_lo}, {pos_hi}) holds {r1 - r0} rows")
    _check_tensor(k_shard, "k_shard", bf, (B, H, rows, d), dev)
    _check_tensor(v_shard, "v_shard", bf, (B, H, rows, d), dev)
    _check_tensor(q, "q", bf, (B, H, d), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", bf, (H, d), dev)
        _check_tensor(v0, "v0", bf, (H, d), dev)
    else:
        k0 = v0 = None
    if seqlens is not None:
        _check_tensor(seqlens, "seqlens", torch.int32, (B,), dev)
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    _check_tensor(out, "out", torch.float32, (B, H, d), dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    _check_tensor(lse, "lse", torch.float32, (B, H), dev)
    if workspace is None:
        workspace = torch.empty(max(decode_range_workspace_bytes(B, H, pos_lo, pos_hi, d), 16),
                                dtype=torch.uint8, device=dev)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().csa_decode_range(_ptr(q), _ptr(k_shard), _ptr(v_shard), _ptr(k0), _ptr(v0),
                                   _ptr(seqlens), _ptr(out), _ptr(lse), _ptr(workspace), nbytes,
                                   B, H, int(T), d, float(scale), int(mode), int(pos_lo),
                                   int(pos_hi), _stream_handle(stream)), "csa_decode_range")
    return out, lse


def decode_merge_ranges(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """lse-weighted merge of range partials (csa_decode_merge_ranges).

    o_parts: fp32 CUDA [R, B, H, d]; lse_parts: fp32 [R, B, H].
    Returns (o bf16 [B, H, d], lse fp32 [B, H])."""
    import torch

    R, B, H, d = o_parts.shape
    dev = o_parts.device
    _check_tensor(o_parts, "o_parts", torch.float32, (R, B, H, d), dev)
    _check_tensor(lse_parts, "lse_parts", torch.float32, (R, B, H), dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    _check_tensor(out, "out", torch.bfloat16, (B, H, d), dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    _check_tensor(lse, "lse", torch.float32, (B, H), dev)
    _check(load().csa_decode_merge_ranges(_ptr(o_parts), _ptr(lse_parts), R, B, H, d, _ptr(out),
                                          _ptr(lse), _stream_handle(stream)),
           "csa_decode_merge_ranges")
    return out, lse


def decode_noalloc(q, k_cache, v_cache, k0=None, v0=None, *, seqlens=None, mode: int = 0,
                   scale=None, out=None, lse=None, stream=None, want_lse: bool = True):
    """decode() through csa_decode_noalloc: no workspace, the library's fixed
    device scratch array instead (calls on one device must not overlap)."""
    import torch

    B, H, T, d = k_cache.shape
    dev = k_cache.device
    bf = torch.bfloat16
    _check_tensor(k_cache, "k_cache", bf, (B, H, T, d), dev)
    _check_tensor(v_cache, "v_cache", bf, (B, H, T, d), dev)
    _check_tensor(q, "q", bf, (B, H, d), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", bf, (H, d), dev)
        _check_tensor(v0, "v0", bf, (H, d), dev)
    else:
        k0 = v0 = None
    if seqlens is not None:
        _check_tensor(seqlens, "seqlens", torch.int32, (B,), dev)
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty((B, H, d), dtype=bf, device=dev)
    _check_tensor(out, "out", bf, (B, H, d), dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32, (B, H), dev)
    _check(load().csa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k0), _ptr(v0),
                                     _ptr(seqlens), _ptr(out), _ptr(lse), B, H, T, d,
                                     float(scale), int(mode), _stream_handle(stream)),
           "csa_decode_noalloc")
    return out, lse


def backward_workspace_bytes(B: int, H: int, T: int, d: int) -> int:
    """Bytes of workspace csa_backward needs (host-side, no device needed)."""
    n = int(load().csa_backward_workspace_bytes(int(B), int(H), int(T), int(d)))
    if n < 0:
        raise CsaError(CSA_ERR_UNSUPPORTED, "csa_backward_workspace_bytes")
    return n


def backward(q, k, v, out, lse, dout, k0=None, v0=None, *, mode: int = 0, scale=None,
             dq=None, dk=None, dv=None, dk0=None, dv0=None, workspace=None, stream=None):
    """Gradients of the continuous forward pass for the upstream gradient
    dout.  q, k, v, out, dout: CUDA [B, H, T, d], all bf16 or all fp32; lse:
    float32 [B, H, T] from forward().  Returns (dq, dk, dv, dk0, dv0); dk0 and
    dv0 (float32 [H, d]) are None unless mode is GIVEN (2)."""
    import torch

    B, H, T, d = q.shape
    dtype, dev = q.dtype, q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_tensor(t, name, dtype, (B, H, T, d), dev)
    _check_tensor(lse, "lse", torch.float32, (B, H, T), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", dtype, (H, d), dev)
        _check_tensor(v0, "v0", dtype, (H, d), dev)
        if dk0 is None:
            dk0 = torch.empty((H, d), dtype=torch.float32, device=dev)
        if dv0 is None:
            dv0 = torch.empty((H, d), dtype=torch.float32, device=dev)
        _check_tensor(dk0, "dk0", torch.float32, (H, d), dev)
        _check_tensor(dv0, "dv0", torch.float32, (H, d), dev)
    else:
        k0 = v0 = dk0 = dv0 = None
    if scale is None:
        scale = 1.0 / d ** 0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(t, name, dtype, (B, H, T, d), dev)
    if workspace is None:
        workspace = torch.empty(max(backward_workspace_bytes(B, H, T, d), 16), dtype=torch.uint8,
                                device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    nbytes = workspace.numel() * workspace.element_size()
    lib = load()
    if dtype == torch.bfloat16:
        fn, where = lib.csa_backward, "csa_backward"
    elif dtype == torch.float32:
        fn, where = lib.csa_backward_f32, "csa_backward_f32"
    else:
        raise ValueError(f"unsupported dtype {dtype}")
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(out), _ptr(lse), _ptr(dout),
              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dk0), _ptr(dv0), _ptr(workspace), nbytes, B, H,
              T, d, float(scale), int(mode), _stream_handle(stream)), where)
    return dq, dk, dv, dk0, dv0


def logphi2_eval(x, stream=None):
    """log phi2 of a float32 CUDA tensor, by the library's device function."""
    import torch

    x = x.contiguous()
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be a float32 CUDA tensor")
    y = torch.empty_like(x)
    _check(load().csa_logphi2_eval(_ptr(x), _ptr(y), x.numel(), _stream_handle(stream)),
           "csa_logphi2_eval")
    return y


def segment_weights_eval(u0, u1, stream=None):
    """(right, left) end weights of intervals (u0 -> u1), tensor-core kernel math."""
    import torch

    u0, u1 = u0.contiguous(), u1.contiguous()
    r = torch.empty_like(u0)
    l_ = torch.empty_like(u0)
    _check(load().csa_segment_weights_eval(_ptr(u0), _ptr(u1), _ptr(r), _ptr(l_), u0.numel(),
                                           _stream_handle(stream)), "csa_segment_weights_eval")
    return r, l_


def device_status() -> int:
    """Reads and clears the library's device status word (synchronises)."""
    return int(load().csa_device_status())


def selftest_forward_delay(q, k, v, k0=None, v0=None, *, mode: int = 0, scale=None,
                           delay_ns: int = 20000, delay_half: int = 1, stream=None):
    """csa_forward's exact form (bf16, d in {64, 128}) with a delay planted
    before each epilogue's reads of the accumulators, for one column half
    (csa_selftest_forward_delay).  Returns (o, lse), which must equal
    forward()'s bit for bit."""
    import torch

    B, H, T, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, name, torch.bfloat16, (B, H, T, d), dev)
    if mode == 2:
        if k0 is None or v0 is None:
            raise ValueError("mode 2 (given sink) needs k0 and v0")
        _check_tensor(k0, "k0", torch.bfloat16, (H, d), dev)
        _check_tensor(v0, "v0", torch.bfloat16, (H, d), dev)
    else:
        k0 = v0 = None
    if scale is None:
        scale = 1.0 / d ** 0.5
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    _check(load().csa_selftest_forward_delay(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(out), _ptr(lse), B, H, T, d,
        float(scale), int(mode), int(delay_ns), int(delay_half), _stream_handle(stream)),
        "csa_selftest_forward_delay")
    return out, lse


def selftest_wait_timeout(timeout_us: int, stream=None):
    _check(load().csa_selftest_wait_timeout(int(timeout_us), _stream_handle(stream)),
           "csa_selftest_wait_timeout")
