"""Chunk-parallel (WY / UT) form of the gated delta rule, fp64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It is a second,
independent statement of the method in the pages' chunked shape, used to
check the GPU's intermediate stages one at a time:

* the sequence of one (sequence, head) unit is cut into fixed tiles of
  ``chunk`` tokens, restarting at the sequence start; work inside a tile is
  parallel and the state is carried from tile to tile by a recursion
  [P1 §3.2, P2 §2.1, P3 §3.1];
* the log-decay is the bounded scaled sigmoid, or the unbounded negative
  softplus it replaces [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3];
* inside a tile every causal block is a dense product once the decays are
  expressed relative to the tile [P1 §3.3, P2 §2.3, P3 §3.3].

Per tile with inclusive in-tile cumulative log-decay G (G_i = sum_{r<=i} g_r),
entering state H0 (dk x dv) and tile length C:

  A_ij = beta_i * exp(G_i - G_j) * (k_i . k_j)    for j < i, else 0
  T    = (I + A)^{-1}                              (unit lower triangular)
  W    = T diag(beta * exp(G)) K                   (C x dk)
  U    = T diag(beta) V                            (C x dv)
  D    = U - W H0                                  (the delta-rule writes)
  O    = diag(exp(G)) Q H0 + (Q K^T (.) M (.) exp(G_i - G_j)) D,  M_ij = [j <= i]
  H1   = exp(G_C) H0 + (K (.) exp(G_C - G))^T D

The triangular inverse uses scipy's triangular solver (a library routine).
Every function is a plain transcription of these definitions: no blocking,
fusion or reordering beyond them.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg
import scipy.special


def gate(a, b: float = 2.0, mode: str = "bounded"):
    """g = -b * sigmoid(a)  or  g = -softplus(a), elementwise, fp64."""
    a = np.asarray(a, dtype=np.float64)
    if mode == "softplus":
        return -np.logaddexp(0.0, a)
    return -b * scipy.special.expit(a)


def tile_cumsum(g, chunk: int):
    """Inclusive cumulative sum of g restarted every ``chunk`` tokens (one unit)."""
    g = np.asarray(g, dtype=np.float64)
    G = np.empty_like(g)
    for s in range(0, g.shape[0], chunk):
        G[s:s + chunk] = np.cumsum(g[s:s + chunk])
    return G


def tile_wy(k, v, beta, G):
    """A, T, W, U of one tile (k [C,dk], v [C,dv], beta [C], G [C])."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64)
    G = np.asarray(G, np.float64)
    C = k.shape[0]
    A = np.tril(beta[:, None] * np.exp(G[:, None] - G[None, :]) * (k @ k.T), -1)
    T = scipy.linalg.solve_triangular(np.eye(C) + A, np.eye(C), lower=True,
                                      unit_diagonal=True)
    W = T @ ((beta * np.exp(G))[:, None] * k)
    U = T @ (beta[:, None] * v)
    return A, T, W, U


def unit_wy(k, v, beta, g, chunk: int):
    """W [L,dk] and U [L,dv] of a whole unit, tile by tile."""
    L = k.shape[0]
    G = tile_cumsum(g, chunk)
    W = np.zeros((L, k.shape[1]))
    U = np.zeros((L, v.shape[1]))
    for s in range(0, L, chunk):
        e = min(s + chunk, L)
        _, _, W[s:e], U[s:e] = tile_wy(k[s:e], v[s:e], beta[s:e], G[s:e])
    return W, U


def unit_fwd(q, k, v, g, beta, h0, chunk: int, record_states: bool = False):
    """Chunked forward of one unit.  Returns (o [L,dv], hT [dk,dv][, states])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64)
    L = q.shape[0]
    H = np.array(h0, dtype=np.float64, copy=True)
    G = tile_cumsum(g, chunk)
    o = np.zeros((L, v.shape[1]))
    states = []
    for s in range(0, L, chunk):
        e = min(s + chunk, L)
        Gc = G[s:e]
        _, _, W, U = tile_wy(k[s:e], v[s:e], beta[s:e], Gc)
        if record_states:
            states.append(H.copy())
        D = U - W @ H
        C = e - s
        mask = np.tril(np.ones((C, C)))
        P = (q[s:e] @ k[s:e].T) * mask * np.exp(Gc[:, None] - Gc[None, :])
        o[s:e] = np.exp(Gc)[:, None] * (q[s:e] @ H) + P @ D
        H = np.exp(Gc[-1]) * H + (k[s:e] * np.exp(Gc[-1] - Gc)[:, None]).T @ D
    if record_states:
        return o, H, states
    return o, H


def fwd(q, k, v, a, beta, h0=None, cu_seqlens=None, chunk: int = 16,
        b: float = 2.0, mode: str = "bounded"):
    """Chunked fp64 forward over the library's layouts (small sizes only)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    a = np.asarray(a, np.float64)
    beta = np.asarray(beta, np.float64)
    B, T, Hh, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(n, n * T, (n + 1) * T) for n in range(B)]
        flat = lambda x: x.reshape((B * T,) + x.shape[2:])  # noqa: E731
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(n, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
        flat = lambda x: x.reshape((T,) + x.shape[2:])  # noqa: E731
    qf, kf, vf, af, bf = (flat(x) for x in (q, k, v, a, beta))
    out = np.zeros((qf.shape[0], Hh, dv))
    hT = np.zeros((len(spans), Hh, dk, dv))
    for n, s, e in spans:
        for h in range(Hh):
            H0 = np.zeros((dk, dv)) if h0 is None else np.asarray(h0, np.float64)[n, h]
            g = gate(af[s:e, h], b, mode)
            o, Hn = unit_fwd(qf[s:e, h], kf[s:e, h], vf[s:e, h], g, bf[s:e, h], H0, chunk)
            out[s:e, h] = o
            hT[n, h] = Hn
    return out.reshape(q.shape[:3] + (dv,)), hT
