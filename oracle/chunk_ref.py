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


# ---------------------------------------------------------------------------
# The backward pass in the same chunked form, with a log-decay per key channel
# (a scalar gate is every channel equal).  The pages print no backward; this is
# the adjoint of the tile algebra above written in its factored form, with
# G [C, dk] the in-tile cumulative log-decay of every channel:
#
#   Kt = K (.) e^G,  Kh = K (.) e^-G,  Qt = Q (.) e^G,  Ke = Kh (.) e^{G_C}
#   A = beta (.) strict_lower(Kt Kh^T),  S = lower(Qt Kh^T),  T = (I + A)^{-1}
#   W = T diag(beta) Kt,  U = T diag(beta) V,  D = U - W H0
#   O = Qt H0 + S D,  H1 = diag(e^{G_C}) H0 + Ke^T D
#
# For L = <dO, O> + <dH_T, H_T> and dH1 the gradient at the tile's end:
#   dD = S^T dO + Ke dH1,   dH0 = diag(e^{G_C}) dH1 + Qt^T dO - W^T dD
#   dS = lower(dO D^T),  dKe = D dH1^T,  dW = -dD H0^T,  dQt = dO H0^T + dS Kh
#   dYu = T^T dD,  dYw = T^T dW,  dA = -strict_lower(dYu U^T + dYw W^T)
#   dV = diag(beta) dYu,  dKt = diag(beta) dYw + (beta (.) dA) Kh
#   dKh = (beta (.) dA)^T Kt + dS^T Qt + dKe (.) e^{G_C}
#   dbeta_i = dYu_i . V_i + dYw_i . Kt_i + sum_j dA_ij (Kt Kh^T)_ij
#   dG = dQt (.) Qt + dKt (.) Kt - dKh (.) Kh, and at the last token also
#        sum_i dKe_i (.) Ke_i + e^{G_C} (.) rowsum(dH1 (.) H0)
#   dg = the reverse cumulative sum of dG inside the tile
#   dq = dQt (.) e^G,  dk = dKt (.) e^G + dKh (.) e^-G
# It is checked against the token-by-token adjoint of the C oracle, which is
# pinned by finite differences.
# ---------------------------------------------------------------------------
def gate_grad(a, b: float = 2.0, mode: str = "bounded"):
    """dg/da elementwise, fp64: -b sigmoid (1 - sigmoid), or -sigmoid for softplus."""
    s = scipy.special.expit(np.asarray(a, dtype=np.float64))
    if mode == "softplus":
        return -s
    return -b * s * (1.0 - s)


def _tile_channels(q, k, v, g, beta, H0):
    """Forward quantities of one tile with per-channel log-decays g [C, dk]."""
    C = k.shape[0]
    G = np.cumsum(g, axis=0)
    eG, enG = np.exp(G), np.exp(-G)
    Kt, Kh, Qt = k * eG, k * enG, q * eG
    eGC = eG[-1]
    Ke = Kh * eGC
    A = beta[:, None] * np.tril(Kt @ Kh.T, -1)
    S = np.tril(Qt @ Kh.T)
    T = scipy.linalg.solve_triangular(np.eye(C) + A, np.eye(C), lower=True, unit_diagonal=True)
    W = T @ (beta[:, None] * Kt)
    U = T @ (beta[:, None] * v)
    D = U - W @ H0
    H1 = eGC[:, None] * H0 + Ke.T @ D
    O = Qt @ H0 + S @ D
    return dict(G=G, eG=eG, enG=enG, Kt=Kt, Kh=Kh, Qt=Qt, eGC=eGC, Ke=Ke, A=A, S=S, T=T, W=W,
                U=U, D=D, H0=H0, H1=H1, O=O)


def fwd_channels(q, k, v, a, beta, h0=None, cu_seqlens=None, chunk: int = 16, b: float = 2.0,
                 mode: str = "bounded"):
    """Chunked fp64 forward with a log-decay per key channel (a [B,T,H,dk]), tile by
    tile in the factored form above: O = Qt H0 + S D, H1 = diag(e^{G_C}) H0 + Ke^T D.
    Returns (out [B,T,H,dv], hT [N,H,dk,dv]); small sizes only."""
    q, k, v, a, beta = (np.asarray(x, np.float64) for x in (q, k, v, a, beta))
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
            H = np.zeros((dk, dv)) if h0 is None else np.array(h0, np.float64)[n, h]
            g = gate(af[s:e, h], b, mode)
            for t0 in range(s, e, chunk):
                t1 = min(t0 + chunk, e)
                t = _tile_channels(qf[t0:t1, h], kf[t0:t1, h], vf[t0:t1, h], g[t0 - s:t1 - s],
                                   bf[t0:t1, h], H)
                out[t0:t1, h] = t["O"]
                H = t["H1"]
            hT[n, h] = H
    return out.reshape(q.shape[:3] + (dv,)), hT


def tile_grads(t, v, beta, dO, dH1):
    """The gradients of one tile from its forward quantities t (``_tile_channels``),
    its V and beta, the output gradient dO and the gradient dH1 at the tile's end.
    Returns dq, dk [C,dk], dv [C,dv], dg [C,dk], dbeta [C] and dH0 [dk,dv]."""
    dD = t["S"].T @ dO + t["Ke"] @ dH1
    dH0 = t["eGC"][:, None] * dH1 + t["Qt"].T @ dO - t["W"].T @ dD
    dS = np.tril(dO @ t["D"].T)
    dKe = t["D"] @ dH1.T
    dW = -dD @ t["H0"].T
    dQt = dO @ t["H0"].T + dS @ t["Kh"]
    dYu = t["T"].T @ dD
    dYw = t["T"].T @ dW
    dA = -np.tril(dYu @ t["U"].T + dYw @ t["W"].T, -1)
    bdA = beta[:, None] * dA
    dKt = beta[:, None] * dYw + bdA @ t["Kh"]
    dKh = bdA.T @ t["Kt"] + dS.T @ t["Qt"] + dKe * t["eGC"]
    dv = beta[:, None] * dYu
    dbeta = (dYu * v).sum(1) + (dYw * t["Kt"]).sum(1) + (dA * (t["Kt"] @ t["Kh"].T)).sum(1)
    dG = dQt * t["Qt"] + dKt * t["Kt"] - dKh * t["Kh"]
    dG[-1] += (dKe * t["Ke"]).sum(0) + t["eGC"] * (dH1 * t["H0"]).sum(1)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    return dQt * t["eG"], dKt * t["eG"] + dKh * t["enG"], dv, dg, dbeta, dH0


def unit_bwd_channels(q, k, v, g, beta, h0, dout, dhT, chunk: int):
    """Chunked backward of one unit: q, k [L,dk], v [L,dv], g [L,dk], beta [L], h0 and
    dhT [dk,dv], dout [L,dv].  Returns dq, dk [L,dk], dv [L,dv], dg [L,dk], dbeta [L]
    and dh0 [dk,dv]."""
    L = k.shape[0]
    starts = list(range(0, L, chunk))
    tiles, H = [], np.array(h0, dtype=np.float64, copy=True)
    for s in starts:
        e = min(s + chunk, L)
        t = _tile_channels(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], H)
        tiles.append(t)
        H = t["H1"]
    dq, dk_, dg = np.zeros_like(k), np.zeros_like(k), np.zeros_like(k)
    dv_, dbeta = np.zeros_like(v), np.zeros_like(beta)
    dH = np.array(dhT, dtype=np.float64, copy=True)
    for s, t in zip(reversed(starts), reversed(tiles)):
        e = min(s + chunk, L)
        dq[s:e], dk_[s:e], dv_[s:e], dg[s:e], dbeta[s:e], dH = tile_grads(t, v[s:e], beta[s:e],
                                                                          dout[s:e], dH)
    return dq, dk_, dv_, dg, dbeta, dH


def bwd(q, k, v, a, beta, dout=None, dhT=None, h0=None, cu_seqlens=None, chunk: int = 16,
        b: float = 2.0, mode: str = "bounded", per_channel: bool = False):
    """Chunked fp64 backward over the library's layouts (small sizes only), as a dict
    with dq, dk, dv, da, dbeta, dh0 shaped like the oracle's.  a is [B,T,H] (every
    channel shares the gate, da sums its channels' gradients) or, with per_channel,
    [B,T,H,dk]."""
    q, k, v, a, beta = (np.asarray(x, np.float64) for x in (q, k, v, a, beta))
    B, T, Hh, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(n, n * T, (n + 1) * T) for n in range(B)]
        flat = lambda x: x.reshape((B * T,) + x.shape[2:])  # noqa: E731
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(n, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
        flat = lambda x: x.reshape((T,) + x.shape[2:])  # noqa: E731
    dout = np.zeros(v.shape) if dout is None else np.asarray(dout, np.float64)
    qf, kf, vf, af, bf, df = (flat(x) for x in (q, k, v, a, beta, dout))
    rows = qf.shape[0]
    res = dict(dq=np.zeros((rows, Hh, dk)), dk=np.zeros((rows, Hh, dk)), dv=np.zeros((rows, Hh, dv)),
               da=np.zeros(af.shape), dbeta=np.zeros((rows, Hh)),
               dh0=np.zeros((len(spans), Hh, dk, dv)))
    for n, s, e in spans:
        for h in range(Hh):
            H0 = np.zeros((dk, dv)) if h0 is None else np.asarray(h0, np.float64)[n, h]
            dHT = np.zeros((dk, dv)) if dhT is None else np.asarray(dhT, np.float64)[n, h]
            ah = af[s:e, h] if per_channel else np.repeat(af[s:e, h][:, None], dk, axis=1)
            g = gate(ah, b, mode)
            gq, gk, gv, gg, gb, gh = unit_bwd_channels(qf[s:e, h], kf[s:e, h], vf[s:e, h], g,
                                                       bf[s:e, h], H0, df[s:e, h], dHT, chunk)
            res["dq"][s:e, h], res["dk"][s:e, h], res["dv"][s:e, h] = gq, gk, gv
            res["dbeta"][s:e, h], res["dh0"][n, h] = gb, gh
            da = gg * gate_grad(ah, b, mode)
            res["da"][s:e, h] = da if per_channel else da.sum(1)
    shape = q.shape[:3]
    return dict(dq=res["dq"].reshape(shape + (dk,)), dk=res["dk"].reshape(shape + (dk,)),
                dv=res["dv"].reshape(shape + (dv,)), da=res["da"].reshape(a.shape),
                dbeta=res["dbeta"].reshape(shape), dh0=res["dh0"])
