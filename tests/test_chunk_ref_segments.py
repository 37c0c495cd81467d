"""The tensor-core forward's segment scan, restated in fp64 on the chunk form (CPU only).

The sequence's tiles are cut into segments.  Every segment but the last gets a
transition H_out = M H_in + B: B from a zero entering state, M the product of the
tiles' linear maps H -> e^{G_C} H - Ke^T W H.  The transition pass starts at the
first tile r whose accumulated log-decay to the segment's end is <= -64 ln 2; then
M is taken as zero and B starts from zero at r.  If no such r exists, the whole
segment is used.  A serial combine gives every segment's entering state, and an
output pass runs each segment from it.  For unit keys and beta in [0, 1] the
truncated terms are below 2^-64 of the state, so in fp64 the scheme equals the
token-by-token oracle to rounding.  A horizon far too short does not.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import chunk_ref
from test_oracle_pins import _case

TRUNC = 64 * math.log(2.0)


def _tile(q, k, v, g, beta, H):
    """One tile of the chunk form: returns (o, H1, M_tile, B_tile)."""
    G = np.cumsum(g)
    _, _, W, U = chunk_ref.tile_wy(k, v, beta, G)
    C = len(g)
    Ke = k * np.exp(G[-1] - G)[:, None]
    mask = np.tril(np.ones((C, C)))
    P = (q @ k.T) * mask * np.exp(G[:, None] - G[None, :])
    D = U - W @ H
    o = np.exp(G)[:, None] * (q @ H) + P @ D
    M = np.exp(G[-1]) * np.eye(k.shape[1]) - Ke.T @ W
    return o, np.exp(G[-1]) * H + Ke.T @ D, M, Ke.T @ U


def _segment_scan(q, k, v, g, beta, h0, seg_tiles, chunk=16, horizon=TRUNC, erase=True):
    """``erase``: the horizon's bound carries each token's erase-factor norm
    max(1, |1 - beta |k|^2|) beside its decay (the norm of alpha (I - beta k k^T));
    without it the bound is the decay alone, which holds only for 0 <= beta |k|^2 <= 2."""
    L, dk = k.shape
    n_t = (L + chunk - 1) // chunk
    tl = [(c * chunk, min(L, (c + 1) * chunk)) for c in range(n_t)]
    segs = [list(range(s, min(n_t, s + seg_tiles))) for s in range(0, n_t, seg_tiles)]
    log_erase = np.log(np.maximum(1.0, np.abs(1.0 - beta * (k * k).sum(axis=1))))
    Ms, Bs, truncated = [], [], 0
    for seg in segs[:-1]:
        acc, r = 0.0, None
        for c in reversed(seg):
            acc += g[tl[c][0]:tl[c][1]].sum()
            if erase:
                acc += log_erase[tl[c][0]:tl[c][1]].sum()
            if acc <= -horizon:
                r = c
                break
        first = seg[0] if r is None else r
        M, B = np.eye(dk), np.zeros((dk, v.shape[1]))
        for c in range(first, seg[-1] + 1):
            s, e = tl[c]
            _, B, Mt, _ = _tile(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], B)
            M = Mt @ M
        if r is not None:
            M = np.zeros_like(M)
            truncated += 1
        Ms.append(M)
        Bs.append(B)
    H = h0.copy()
    out = np.zeros((L, v.shape[1]))
    for j, seg in enumerate(segs):
        Hs = H
        for c in seg:
            s, e = tl[c]
            out[s:e], Hs, _, _ = _tile(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], Hs)
        if j < len(segs) - 1:
            H = Ms[j] @ H + Bs[j]
        else:
            H = Hs
    return out, H, truncated


def _unit(rng, L, a_mean):
    q, k, v, a, beta, h0 = _case(rng, L, dk=8, dv=6, h0_std=1.0)
    a = a + a_mean
    g = chunk_ref.gate(a[0, :, 0], 2.0)
    return q, k, v, a, beta, h0, g


@pytest.mark.parametrize("a_mean,expect_truncated", [(0.0, True), (-6.0, False)])
def test_segment_scan_equals_the_oracle(a_mean, expect_truncated):
    """a ~ N(0, 1), about 1 of log-decay per token: the horizon lies about three tiles
    before each segment's end, so every transition is truncated.  a ~ N(-6, 1): the
    decay is too weak for the horizon within an 8-tile segment, so the transitions are
    full."""
    rng = np.random.default_rng(400)
    L = 16 * 40
    q, k, v, a, beta, h0, g = _unit(rng, L, a_mean)
    out, hT, trunc = _segment_scan(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0], 8)
    assert (trunc == 4) == expect_truncated and (trunc == 0) == (not expect_truncated)
    ro, rh = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    scale = max(np.abs(ro).max(), 1.0)
    np.testing.assert_allclose(out, ro[0, :, 0], rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(hT, rh[0, 0], rtol=0, atol=1e-12 * max(np.abs(rh).max(), 1.0))


def test_a_short_horizon_is_visible():
    """Truncating at 5 of log-decay instead of 64 ln 2 drops terms of order e^-5 of the
    state, far above fp64 rounding.  The decay is weak (a ~ N(-3, 1), about 1.5 of
    log-decay per tile), so the short horizon truncates several tiles into each segment,
    where the full one would truncate none."""
    rng = np.random.default_rng(401)
    q, k, v, a, beta, h0, g = _unit(rng, 16 * 40, -3.0)
    assert _segment_scan(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0], 8)[2] == 0
    out, _, trunc = _segment_scan(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0], 8,
                                  horizon=5.0)
    assert trunc == 4
    ro, _ = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    assert np.abs(out - ro[0, :, 0]).max() > 1e-6 * np.abs(ro).max()


def _aligned(rng, L, scale, a_mean, a_std):
    """Every key along one direction e_1 with |k|^2 = scale^2, beta = 1: the state's
    e_1 row is multiplied by alpha (1 - scale^2) per token, the rest by alpha."""
    q, k, v, a, beta, h0 = _case(rng, L, dk=8, dv=6, h0_std=1.0)
    k = np.zeros_like(k)
    k[..., 0] = scale
    beta = np.ones_like(beta)
    a = a_mean + a_std * rng.standard_normal(a.shape)
    g = chunk_ref.gate(a[0, :, 0], 2.0)
    return q, k, v, a, beta, h0, g


def test_expansive_erase_factors_need_the_erase_term_in_the_horizon():
    """Aligned keys with beta |k|^2 = 3 (erase-factor norm 2) and g about -0.713 per
    token (alpha about 0.49): the e_1 row of the state shrinks by only ~0.98 per
    token.  The decay alone reaches 64 ln 2 about 62 tokens before each segment's
    end, so a decay-only horizon truncates every transition and drops a state that
    has shrunk to ~0.3 of its size: visibly wrong.  With the erase term the bound
    never falls inside a 16-tile segment, no transition is truncated, and the scan
    equals the oracle to rounding."""
    rng = np.random.default_rng(402)
    L = 16 * 16 * 5
    q, k, v, a, beta, h0, g = _aligned(rng, L, math.sqrt(3.0), -0.59, 0.02)
    args = (q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0], 16)
    ro, rh = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    out, hT, trunc = _segment_scan(*args)
    assert trunc == 0
    np.testing.assert_allclose(out, ro[0, :, 0], rtol=0, atol=1e-11 * np.abs(ro).max())
    np.testing.assert_allclose(hT, rh[0, 0], rtol=0, atol=1e-11 * np.abs(rh).max())
    out_d, hT_d, trunc_d = _segment_scan(*args, erase=False)
    assert trunc_d == 4
    rel = np.linalg.norm(out_d - ro[0, :, 0]) / np.linalg.norm(ro)
    assert rel > 0.05, rel


def test_erase_term_still_truncates_non_unit_random_keys():
    """Random keys scaled to |k| = 1.5 with beta in (0, 1) (beta |k|^2 up to 2.25) and
    a ~ N(0, 1): the erase term lengthens the horizon a little but every transition is
    still truncated, and the scan equals the oracle to rounding."""
    rng = np.random.default_rng(403)
    L = 16 * 40
    q, k, v, a, beta, h0, g = _unit(rng, L, 0.0)
    k = 1.5 * k
    out, hT, trunc = _segment_scan(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0], 8)
    assert trunc == 4
    ro, rh = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    np.testing.assert_allclose(out, ro[0, :, 0], rtol=0, atol=1e-12 * max(np.abs(ro).max(), 1.0))
    np.testing.assert_allclose(hT, rh[0, 0], rtol=0, atol=1e-12 * max(np.abs(rh).max(), 1.0))
