"""Eq. (2) evaluated by numerical quadrature (test infrastructure only).

Jianlin Su, "Continuous Softmax Attention", section "Problem Statement":
eq. (2) defines o_t as the ratio of two integrals over s in [0, t], with k_s
and v_s linearly interpolated between integer points by eq. (3) and the extra
k_0, v_0 covering s in [0, 1].

This module integrates those definitions directly: on every unit interval
[i-1, i] it interpolates k_s and v_s from the two end vectors, forms
q_t . k_s, and applies composite Gauss-Legendre quadrature.  No phi function
and none of the closed forms (4)-(11) appear here, which is what makes it an
independent check of the closed-form oracle.  The Gauss-Legendre nodes come
from numpy's ``leggauss``.

Each unit interval is split into ``ceil(|delta|/2)`` equal pieces (delta the
change of the logit across the interval), each with ``nodes`` points, so the
exponential never varies by more than e^2 inside one piece and the rule stays
accurate to ~1e-14 for the tiny shapes it is used on.
"""
from __future__ import annotations

import math

import numpy as np

ZERO, COPY_FIRST, GIVEN = 0, 1, 2


def _extended(k, v, k0, v0, h, mode):
    """Rows 0..T of the extended sequence: index 0 is the sink (k_0, v_0)."""
    d = k.shape[-1]
    if mode == ZERO:
        s_k, s_v = np.zeros(d), np.zeros(d)
    elif mode == COPY_FIRST:
        s_k, s_v = k[0], v[0]
    elif mode == GIVEN:
        s_k, s_v = k0[h], v0[h]
    else:
        raise ValueError("mode")
    return np.vstack([s_k[None], k]), np.vstack([s_v[None], v])


def forward(q, k, v, k0=None, v0=None, scale=None, mode=ZERO, nodes=20):
    """o and lse of eq. (2) by quadrature; lse_t = log of eq. (2)'s denominator.

    q, k, v: arrays [B, H, T, d] (converted to float64); k0, v0: [H, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if mode == GIVEN:
        k0 = np.asarray(k0, dtype=np.float64)
        v0 = np.asarray(v0, dtype=np.float64)
    xg, wg = np.polynomial.legendre.leggauss(nodes)
    xi_unit = 0.5 * (xg + 1.0)  # nodes mapped to [0, 1]
    w_unit = 0.5 * wg
    out = np.zeros((B, H, T, d))
    lse = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            K, V = _extended(k[b, h], v[b, h], k0, v0, h, mode)
            for r in range(T):
                t = r + 1
                qt = q[b, h, r]
                # Gather every quadrature point of [0, t].
                pts_logit, pts_val, pts_w = [], [], []
                for i in range(1, t + 1):
                    # logit change across the interval, only to choose the split
                    delta = scale * (qt @ (K[i] - K[i - 1]))
                    pieces = max(1, int(math.ceil(abs(delta) / 2.0)))
                    for p in range(pieces):
                        s_loc = (p + xi_unit) / pieces  # position inside [i-1, i], in [0,1]
                        # eq. (3): k_s = (i - s) k_{i-1} + (s - i + 1) k_i with s = i-1+s_loc
                        ks = np.outer(1.0 - s_loc, K[i - 1]) + np.outer(s_loc, K[i])
                        vs = np.outer(1.0 - s_loc, V[i - 1]) + np.outer(s_loc, V[i])
                        pts_logit.append(scale * (ks @ qt))
                        pts_val.append(vs)
                        pts_w.append(w_unit / pieces)
                lg = np.concatenate(pts_logit)
                vv = np.concatenate(pts_val)
                ww = np.concatenate(pts_w)
                m = lg.max()
                e = ww * np.exp(lg - m)
                den = e.sum()
                out[b, h, r] = (e[:, None] * vv).sum(axis=0) / den
                lse[b, h, r] = m + math.log(den)
    return out, lse


def forward_symmetric(q, k, v, scale=None, nodes=20):
    """The symmetric interval of the original Continuum Attention paper (cited
    in "Problem Statement"): eq. (2)'s integrals over [1/2, t + 1/2] instead of
    [0, t].  Inside [1, t], k_s and v_s follow eq. (3); the end half-cells
    [1/2, 1] and [t, t + 1/2] hold k_1, v_1 and k_t, v_t constant (a causal
    row has no k_{t+1}), so no sink is needed.  By quadrature, as forward()."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    xg, wg = np.polynomial.legendre.leggauss(nodes)
    xi_unit = 0.5 * (xg + 1.0)
    w_unit = 0.5 * wg
    out = np.zeros((B, H, T, d))
    lse = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            K, V = k[b, h], v[b, h]  # row j is the page's key j + 1
            for r in range(T):
                t = r + 1
                qt = q[b, h, r]
                pts_logit, pts_val, pts_w = [], [], []
                # half-cells: a constant integrand over a length of 1/2 each
                for j in {0, t - 1}:
                    pts_logit.append(np.full(nodes, scale * (K[j] @ qt)))
                    pts_val.append(np.tile(V[j], (nodes, 1)))
                    pts_w.append(w_unit * (0.5 if t > 1 else 1.0))
                # eq. (3) on the unit intervals [i-1, i], i = 2..t (page keys)
                for i in range(2, t + 1):
                    a0, a1 = K[i - 2], K[i - 1]
                    delta = scale * (qt @ (a1 - a0))
                    pieces = max(1, int(math.ceil(abs(delta) / 2.0)))
                    for p in range(pieces):
                        s_loc = (p + xi_unit) / pieces
                        ks = np.outer(1.0 - s_loc, a0) + np.outer(s_loc, a1)
                        vs = np.outer(1.0 - s_loc, V[i - 2]) + np.outer(s_loc, V[i - 1])
                        pts_logit.append(scale * (ks @ qt))
                        pts_val.append(vs)
                        pts_w.append(w_unit / pieces)
                lg = np.concatenate(pts_logit)
                vv = np.concatenate(pts_val)
                ww = np.concatenate(pts_w)
                m = lg.max()
                e = ww * np.exp(lg - m)
                den = e.sum()
                out[b, h, r] = (e[:, None] * vv).sum(axis=0) / den
                lse[b, h, r] = m + math.log(den)
    return out, lse
