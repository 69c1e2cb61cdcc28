"""CPU oracle for Continuous Softmax Attention (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The CUDA library and its Python binding never import it, and it shares no
code, header, table or helper with them.

What it computes follows Jianlin Su, "Continuous Softmax Attention"
(Scientific Spaces #11980):

* ``forward``        - eq. (8), the segment sum of the integrals (4)/(5);
                       this is the primary oracle.
* ``forward_eq11``   - eq. (10)/(11), the softmax of ``a + b``.
* ``forward_rows``   - eq. (8) for selected rows only (large shapes).
* ``std_forward``    - eq. (12), standard causal softmax attention.
* ``forward_symmetric`` - eq. (8) over the symmetric interval [1/2, t + 1/2]
                       of the original Continuum Attention paper (constant
                       end half-cells, no sink).
* ``forward_short_conv`` - the short-conv reading of eq. (13): b replaced by
                       its first-order Taylor term (a cheaper variant).
* ``row_bias``       - the logits ``a`` and corrections ``b`` of eq. (10)
                       for one row.
* ``phi1``/``phi2``/``log_phi1``/``log_phi2`` - eq. (6) and its limits.
* ``backward``       - gradients of eq. (10)/(11) with respect to q, k, v
                       and the trainable sink pair, by the plain chain rule
                       (``csa_oracle_backward.c``); ``log_dphi2`` is
                       log phi2'(x), the derivative it needs.
* ``oracle.quadrature.forward`` - eq. (2) itself by composite Gauss-Legendre
                       quadrature over the linearly interpolated keys and
                       values of eq. (3); it uses no phi function.

Everything is computed in float64 from float32 inputs (bf16 inputs are
passed as their exact float32 values).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH, SOURCES, build_oracle

ZERO, COPY_FIRST, GIVEN = 0, 1, 2

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH) or any(
            os.path.getmtime(LIB_PATH) < os.path.getmtime(src) for src in SOURCES):
        build_oracle()
    lib = ctypes.CDLL(LIB_PATH)
    d = ctypes.c_double
    i = ctypes.c_int
    p = ctypes.c_void_p
    ll = ctypes.c_longlong
    for name in ("csa_oracle_phi1", "csa_oracle_phi2", "csa_oracle_log_phi1", "csa_oracle_log_phi2"):
        f = getattr(lib, name)
        f.restype = d
        f.argtypes = [d]
    common = [p, p, p, p, p, p, p, i, i, i, i, d, i, i]
    lib.csa_oracle_forward.argtypes = common
    lib.csa_oracle_forward.restype = i
    lib.csa_oracle_forward_eq11.argtypes = common
    lib.csa_oracle_forward_eq11.restype = i
    lib.csa_oracle_std_forward.argtypes = [p, p, p, p, p, i, i, i, i, d, i]
    lib.csa_oracle_std_forward.restype = i
    lib.csa_oracle_forward_rows.argtypes = [p, p, p, p, p, p, ll, p, p, i, i, i, i, d, i, i]
    lib.csa_oracle_forward_rows.restype = i
    lib.csa_oracle_std_forward_rows.argtypes = [p, p, p, p, ll, p, p, i, i, i, i, d, i]
    lib.csa_oracle_std_forward_rows.restype = i
    lib.csa_oracle_row_bias.argtypes = [p, p, p, i, i, i, i, d, i, i, i, i, p, p]
    lib.csa_oracle_row_bias.restype = i
    lib.csa_oracle_forward_short_conv.argtypes = common
    lib.csa_oracle_forward_short_conv.restype = i
    lib.csa_oracle_forward_short_conv_rows.argtypes = [p, p, p, p, p, p, ll, p, p, i, i, i, i, d, i, i]
    lib.csa_oracle_forward_short_conv_rows.restype = i
    lib.csa_oracle_forward_symmetric.argtypes = [p, p, p, p, p, i, i, i, i, d, i]
    lib.csa_oracle_forward_symmetric.restype = i
    lib.csa_oracle_forward_symmetric_rows.argtypes = [p, p, p, p, ll, p, p, i, i, i, i, d, i]
    lib.csa_oracle_forward_symmetric_rows.restype = i
    lib.csa_oracle_log_dphi2.restype = d
    lib.csa_oracle_log_dphi2.argtypes = [d]
    lib.csa_oracle_backward.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i, i, i, i, d, i, i]
    lib.csa_oracle_backward.restype = i
    _lib = lib
    return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shape(q):
    if q.ndim != 4:
        raise ValueError("q must be [B, H, T, d]")
    return q.shape


def phi1(x: float) -> float:
    return _load().csa_oracle_phi1(float(x))


def phi2(x: float) -> float:
    return _load().csa_oracle_phi2(float(x))


def log_phi1(x: float) -> float:
    return _load().csa_oracle_log_phi1(float(x))


def log_phi2(x: float) -> float:
    return _load().csa_oracle_log_phi2(float(x))


def _prep(q, k, v, k0, v0, mode):
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, T, d = _shape(q)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, T, d]")
    if mode == GIVEN:
        k0, v0 = _f32(k0), _f32(v0)
        if k0 is None or v0 is None or k0.shape != (H, d) or v0.shape != (H, d):
            raise ValueError("given k0/v0 must be [H, d]")
    else:
        k0 = v0 = None
    return q, k, v, k0, v0, (B, H, T, d)


def _run(fn, q, k, v, k0, v0, scale, mode, nthreads):
    q, k, v, k0, v0, (B, H, T, d) = _prep(q, k, v, k0, v0, mode)
    out = np.zeros((B, H, T, d), dtype=np.float64)
    lse = np.zeros((B, H, T), dtype=np.float64)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(out), _ptr(lse),
            B, H, T, d, float(scale), int(mode), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def forward(q, k, v, k0=None, v0=None, scale=None, mode=ZERO, nthreads=None):
    """Continuous attention by eq. (8).  Returns (o, lse) as float64 arrays."""
    if scale is None:
        scale = 1.0 / np.sqrt(_f32(q).shape[-1])
    return _run(_load().csa_oracle_forward, q, k, v, k0, v0, scale, mode, nthreads)


def forward_eq11(q, k, v, k0=None, v0=None, scale=None, mode=ZERO, nthreads=None):
    """Continuous attention by eq. (10)/(11).  Returns (o, lse)."""
    if scale is None:
        scale = 1.0 / np.sqrt(_f32(q).shape[-1])
    return _run(_load().csa_oracle_forward_eq11, q, k, v, k0, v0, scale, mode, nthreads)


def forward_short_conv(q, k, v, k0=None, v0=None, scale=None, mode=ZERO, nthreads=None):
    """The short-conv reading of eq. (13): b replaced by its first-order
    Taylor term ((a_{i-1} + a_{i+1} - 2 a_i)/6 inside, -log 2 + step/3 at the
    two ends).  Returns (o, lse)."""
    if scale is None:
        scale = 1.0 / np.sqrt(_f32(q).shape[-1])
    return _run(_load().csa_oracle_forward_short_conv, q, k, v, k0, v0, scale, mode, nthreads)


def forward_short_conv_rows(q, k, v, rows, k0=None, v0=None, scale=None, mode=ZERO,
                            nthreads=None):
    """forward_short_conv for the flat rows given.  Returns (o[nrows, d], lse[nrows])."""
    q, k, v, k0, v0, (B, H, T, d) = _prep(q, k, v, k0, v0, mode)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().csa_oracle_forward_short_conv_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(rows), n, _ptr(out), _ptr(lse), B, H,
        T, d, float(scale), int(mode), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def forward_symmetric(q, k, v, scale=None, nthreads=None):
    """eq. (8) over the symmetric interval [1/2, t + 1/2] (constant end
    half-cells, no sink).  Returns (o, lse)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, T, d = _shape(q)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, H, T, d), dtype=np.float64)
    lse = np.zeros((B, H, T), dtype=np.float64)
    rc = _load().csa_oracle_forward_symmetric(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                              B, H, T, d, float(scale),
                                              int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def forward_symmetric_rows(q, k, v, rows, scale=None, nthreads=None):
    """forward_symmetric for the flat rows given.  Returns (o[nrows, d], lse[nrows])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, T, d = _shape(q)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().csa_oracle_forward_symmetric_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), n,
                                                   _ptr(out), _ptr(lse), B, H, T, d, float(scale),
                                                   int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def std_forward(q, k, v, scale=None, nthreads=None):
    """Standard causal softmax attention, eq. (12).  Returns (o, lse)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, T, d = _shape(q)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, H, T, d), dtype=np.float64)
    lse = np.zeros((B, H, T), dtype=np.float64)
    rc = _load().csa_oracle_std_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                        B, H, T, d, float(scale), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def flat_rows(B, H, T, picks):
    """(b, h, r) triples -> flat row indices (b*H + h)*T + r."""
    return np.asarray([(b * H + h) * T + r for (b, h, r) in picks], dtype=np.int64)


def forward_rows(q, k, v, rows, k0=None, v0=None, scale=None, mode=ZERO, nthreads=None, std=False):
    """eq. (8) (or eq. (12) with ``std=True``) for the flat rows given.

    Returns (o[nrows, d], lse[nrows])."""
    q, k, v, k0, v0, (B, H, T, d) = _prep(q, k, v, k0, v0, mode if not std else ZERO)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    nt = int(nthreads or default_threads())
    lib = _load()
    if std:
        rc = lib.csa_oracle_std_forward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), n, _ptr(out),
                                             _ptr(lse), B, H, T, d, float(scale), nt)
    else:
        rc = lib.csa_oracle_forward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(rows),
                                         n, _ptr(out), _ptr(lse), B, H, T, d, float(scale),
                                         int(mode), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse


def row_bias(q, k, b, h, r, k0=None, scale=None, mode=ZERO):
    """Logits a_{t,0..t} and corrections b_{t,0..t} (eq. (10)) of row r."""
    q, k = _f32(q), _f32(k)
    B, H, T, d = _shape(q)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    k0 = _f32(k0) if mode == GIVEN else None
    a = np.zeros(r + 2, dtype=np.float64)
    bb = np.zeros(r + 2, dtype=np.float64)
    rc = _load().csa_oracle_row_bias(_ptr(q), _ptr(k), _ptr(k0), B, H, T, d, float(scale),
                                     int(mode), int(b), int(h), int(r), _ptr(a), _ptr(bb))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return a, bb


def decode_range(q, k_cache, v_cache, seqlens, pos_lo, pos_hi, k0=None, v0=None, scale=None,
                 mode=ZERO):
    """The decode step restricted to the positions [pos_lo, pos_hi) of each
    row (position 0 the sink, position i >= 1 cache row i - 1): eq. (11) of
    row t = n_b summed over those positions only, each weight e^{a+b} with b
    from both neighbours (eq. (10), via row_bias).

    q: [B, H, d]; k_cache, v_cache: [B, H, T, d]; seqlens: B lengths.
    Returns (o [B, H, d], lse [B, H]) in float64; a row with no position in
    the range gives o = 0 and lse = -inf.  Ranges that partition [0, n_b]
    merge, weighted by e^{lse}, into the whole row's o and lse."""
    q = _f32(q)
    k, v = _f32(k_cache), _f32(v_cache)
    B, H, T, d = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    k0 = _f32(k0) if mode == GIVEN else None
    v0 = _f32(v0) if mode == GIVEN else None
    o = np.zeros((B, H, d), dtype=np.float64)
    lse = np.full((B, H), -np.inf, dtype=np.float64)
    for b in range(B):
        n = int(seqlens[b])
        lo, hi = pos_lo, min(pos_hi, n + 1)
        if lo >= hi:
            continue
        for h in range(H):
            qrow = np.zeros((1, 1, n, d), dtype=np.float32)
            qrow[0, 0, n - 1] = q[b, h]
            kh = np.ascontiguousarray(k[b:b + 1, h:h + 1, :n])
            a, bb = row_bias(qrow, kh, 0, 0, n - 1, k0[h:h + 1] if k0 is not None else None,
                             scale=scale, mode=mode)
            z = (a + bb)[lo:hi]
            m = z.max()
            w = np.exp(z - m)
            if mode == GIVEN:
                sink_v = v0[h].astype(np.float64)
            elif mode == COPY_FIRST:
                sink_v = v[b, h, 0].astype(np.float64)
            else:
                sink_v = np.zeros(d)
            vals = np.vstack([sink_v[None], v[b, h, :n].astype(np.float64)])[lo:hi]
            o[b, h] = (w[:, None] * vals).sum(axis=0) / w.sum()
            lse[b, h] = m + np.log(w.sum())
    return o, lse


def log_dphi2(x: float) -> float:
    """log phi2'(x), phi2'(x) = int_0^1 s (1 - s) e^{sx} ds."""
    return _load().csa_oracle_log_dphi2(float(x))


def backward(q, k, v, dout, k0=None, v0=None, scale=None, mode=ZERO, nthreads=None):
    """Gradients of L = sum(dout * o) for the continuous forward pass.

    Returns dict(dq, dk, dv, dk0, dv0) of float64 arrays ([B, H, T, d], and
    [H, d] for the sink pair in mode GIVEN, else None)."""
    q, k, v, k0, v0, (B, H, T, d) = _prep(q, k, v, k0, v0, mode)
    g = _f32(dout)
    if g.shape != q.shape:
        raise ValueError("dout must be [B, H, T, d]")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros((B, H, T, d), dtype=np.float64)
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    dk0 = np.zeros((H, d), dtype=np.float64) if mode == GIVEN else None
    dv0 = np.zeros((H, d), dtype=np.float64) if mode == GIVEN else None
    rc = _load().csa_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(k0), _ptr(v0), _ptr(g),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dk0), _ptr(dv0),
                                     B, H, T, d, float(scale), int(mode),
                                     int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return {"dq": dq, "dk": dk, "dv": dv, "dk0": dk0, "dv0": dv0}
