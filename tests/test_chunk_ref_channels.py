"""The chunked per-channel forward and backward formulas against the token-by-token
oracle (CPU only).

``oracle.chunk_ref.bwd`` states the backward pass in the chunked, factored form
the GPU's chunked backward computes (per tile: the two state chains' quantities,
the triangular solves by back substitution, the gradients of every input).  The
pages print no backward; this form is the adjoint of the tile algebra.  In fp64 it
must equal the C oracle's token-by-token adjoint recurrence, itself pinned by
finite differences of the forward, to rounding: the chunked form is exact, not an
approximation, so the GPU's tolerance only has to cover its own rounding.
"""
import numpy as np
import pytest

import oracle
from oracle import chunk_ref
from test_oracle_pins import _case

NAMES = ("dq", "dk", "dv", "da", "dbeta", "dh0")


def _grads(rng, B, T, H, dk, dv, per_channel):
    q, k, v, a, beta, h0 = _case(rng, T, H=H, dk=dk, dv=dv, B=B)
    if per_channel:
        a = rng.standard_normal((B, T, H, dk))
    dout = rng.standard_normal(v.shape)
    dhT = 0.1 * rng.standard_normal(h0.shape)
    return q, k, v, a, beta, h0, dout, dhT


def _close(got, ref, rtol=1e-9):
    for n in NAMES:
        scale = max(1.0, float(np.abs(ref[n]).max()))
        err = float(np.abs(got[n] - ref[n]).max())
        assert err <= rtol * scale, f"{n}: max error {err:.3e} (scale {scale:.3e})"


@pytest.mark.parametrize("T,chunk", [(1, 16), (16, 16), (37, 16), (50, 8)])
@pytest.mark.parametrize("per_channel", [False, True])
def test_chunked_backward_equals_token_adjoint(T, chunk, per_channel):
    rng = np.random.default_rng(100 + T + chunk + per_channel)
    q, k, v, a, beta, h0, dout, dhT = _grads(rng, 2, T, 2, 6, 5, per_channel)
    got = chunk_ref.bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, chunk=chunk,
                        per_channel=per_channel)
    fn = oracle.oracle_bwd_vec if per_channel else oracle.oracle_bwd
    ref = fn(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    _close(got, ref)


def test_chunked_backward_packed_sequences_and_large_bound():
    """Packed sequences (one empty) and b = 5, the largest bound the factored
    in-tile form takes at 16-token tiles (e^{-G} up to e^{80})."""
    rng = np.random.default_rng(7)
    q, k, v, a, beta, h0, dout, dhT = _grads(rng, 1, 70, 2, 6, 5, True)
    cu = np.array([0, 9, 9, 40, 70])
    h0 = 0.1 * rng.standard_normal((4, 2, 6, 5))
    dhT = 0.1 * rng.standard_normal((4, 2, 6, 5))
    a = 3.0 * a
    got = chunk_ref.bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, cu_seqlens=cu, b=5.0,
                        per_channel=True)
    ref = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, cu_seqlens=cu, b=5.0)
    _close(got, ref)
    np.testing.assert_array_equal(got["dh0"][1], dhT[1])   # the empty sequence


def test_chunked_backward_without_optional_inputs():
    rng = np.random.default_rng(8)
    q, k, v, a, beta, _, dout, _ = _grads(rng, 1, 30, 1, 4, 3, False)
    got = chunk_ref.bwd(q, k, v, a, beta, dout=dout)
    ref = oracle.oracle_bwd(q, k, v, a, beta, dout=dout, b=2.0)
    _close(got, ref)


def test_a_wrong_tile_term_is_caught():
    """Dropping the last token's e^{G_C} rowsum(dH1 (.) H0) term from dG, the one that
    is easiest to miss, moves da well outside the tolerance."""
    rng = np.random.default_rng(9)
    q, k, v, a, beta, h0, dout, dhT = _grads(rng, 1, 33, 1, 6, 5, True)
    ref = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    saved = chunk_ref.unit_bwd_channels

    def without_state_term(q_, k_, v_, g_, b_, h0_, do_, dh_, chunk):
        out = list(saved(q_, k_, v_, g_, b_, h0_, do_, dh_, chunk))
        # recompute dg with the state term of every tile removed
        L = k_.shape[0]
        H = np.array(h0_, copy=True)
        tiles = []
        for s in range(0, L, chunk):
            t = chunk_ref._tile_channels(q_[s:s + chunk], k_[s:s + chunk], v_[s:s + chunk],
                                         g_[s:s + chunk], b_[s:s + chunk], H)
            tiles.append((s, t))
            H = t["H1"]
        dH = np.array(dh_, copy=True)
        for s, t in reversed(tiles):
            e = min(s + chunk, L)
            dO = do_[s:e]
            dD = t["S"].T @ dO + t["Ke"] @ dH
            out[3][s:e] -= t["eGC"] * (dH * t["H0"]).sum(1)   # the term reaches every dg of the tile
            dH = t["eGC"][:, None] * dH + t["Qt"].T @ dO - t["W"].T @ dD
        return tuple(out)

    chunk_ref.unit_bwd_channels = without_state_term
    try:
        bad = chunk_ref.bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, per_channel=True)
    finally:
        chunk_ref.unit_bwd_channels = saved
    err = float(np.abs(bad["da"] - ref["da"]).max())
    assert err > 1e-3 * max(1.0, float(np.abs(ref["da"]).max()))


@pytest.mark.parametrize("T,chunk,b", [(1, 16, 2.0), (37, 16, 2.0), (64, 16, 5.0), (45, 8, 2.0)])
def test_chunked_per_channel_forward_equals_token_recurrence(T, chunk, b):
    """The factored per-channel tile form of the GPU's per-channel forward (Kt, Kh, Qt,
    Ke, A, S, W, U, D per tile) equals the per-channel oracle to rounding."""
    rng = np.random.default_rng(200 + T + chunk)
    q, k, v, a, beta, h0, _, _ = _grads(rng, 2, T, 2, 6, 5, True)
    o, hT = chunk_ref.fwd_channels(q, k, v, a, beta, h0=h0, chunk=chunk, b=b)
    ro, rh = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=b)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hT, rh, rtol=1e-10, atol=1e-12)


def test_chunked_per_channel_forward_packed_sequences():
    rng = np.random.default_rng(11)
    q, k, v, a, beta, _, _, _ = _grads(rng, 1, 70, 2, 6, 5, True)
    cu = np.array([0, 9, 9, 40, 70])
    h0 = 0.1 * rng.standard_normal((4, 2, 6, 5))
    o, hT = chunk_ref.fwd_channels(q, k, v, a, beta, h0=h0, cu_seqlens=cu)
    ro, rh = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, cu_seqlens=cu, b=2.0)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hT, rh, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(hT[1], h0[1])


# ---- the segment scheme of the per-channel kernels, in fp64 -----------------------------
def _segmented(q, k, v, a, beta, h0, S, b=2.0, erase_term=True, horizon=-46.0, chunk=16):
    """One (sequence, head): q, k [L,dk], v [L,dv], a [L,dk], beta [L].  Tiles are cut
    into segments of S tiles.  Segment j > 0 starts from a zero state at the latest tile
    w <= j S whose bound to j S, sum over its tokens of max_d g + ln max(1, |1 - beta |k|^2|),
    is <= horizon.  w = 0 starts from h0.  If some segment start has no such w within
    4 S tiles, the whole sequence runs as one segment.  Returns (out, hT, warm-ups)."""
    L = q.shape[0]
    g = chunk_ref.gate(a, b)
    n_t = (L + chunk - 1) // chunk
    lam = np.zeros(n_t)
    for c in range(n_t):
        s, e = c * chunk, min(L, (c + 1) * chunk)
        erase = np.log(np.maximum(1.0, np.abs(1.0 - beta[s:e] * (k[s:e] ** 2).sum(1))))
        lam[c] = g[s:e].max(axis=1).sum() + (erase.sum() if erase_term else 0.0)
    starts = list(range(0, n_t, S))
    warm = {}
    for s0 in starts[1:]:
        acc, w = 0.0, None
        for c in range(s0 - 1, max(-1, s0 - 4 * S - 1), -1):
            acc += lam[c]
            if acc <= horizon:
                w = c
                break
        if w is None and s0 > 4 * S:
            starts, warm = [0], {}           # no warm-up: one segment
            break
        warm[s0] = 0 if w is None else w
    out = np.zeros((L, v.shape[1]))
    hT = None
    for j, s0 in enumerate(starts):
        s1 = starts[j + 1] if j + 1 < len(starts) else n_t
        w = warm.get(s0, 0)
        H = h0.copy() if w == 0 else np.zeros_like(h0)
        for c in range(w, s1):
            ts, te = c * chunk, min(L, (c + 1) * chunk)
            t = chunk_ref._tile_channels(q[ts:te], k[ts:te], v[ts:te], g[ts:te], beta[ts:te], H)
            if c >= s0:
                out[ts:te] = t["O"]
            H = t["H1"]
        hT = H
    return out, hT, warm


def _unit(rng, L, dk=8, dv=6, key_scale=1.0):
    q, k, v, _, beta, h0 = _case(rng, L, dk=dk, dv=dv, h0_std=1.0)
    a = rng.standard_normal((1, L, 1, dk))
    return (q[0, :, 0], key_scale * k[0, :, 0], v[0, :, 0], a[0, :, 0], beta[0, :, 0], h0[0, 0])


def test_segments_from_warm_up_tiles_reproduce_the_sequence():
    """Unit keys, a ~ N(0, 1): every segment start finds a warm-up tile after the
    sequence start (7 or 8 tiles back with 8 channels), so every later segment drops its
    earlier history.  The segmented outputs and final state still equal the unsegmented
    oracle to fp64 rounding: the dropped parts are below e^-46 of the state."""
    rng = np.random.default_rng(300)
    q, k, v, a, beta, h0 = _unit(rng, 16 * 48)
    out, hT, warm = _segmented(q, k, v, a, beta, h0, S=8)
    assert len(warm) == 5 and all(0 < w and s0 - w <= 4 * 8 for s0, w in warm.items())   # all truncate
    ro, rh = oracle.oracle_fwd_vec(*(x[None, :, None] for x in (q, k, v, a, beta)), h0=h0[None, None],
                                   b=2.0)
    np.testing.assert_allclose(out, ro[0, :, 0], rtol=0, atol=1e-12 * np.abs(ro).max())
    np.testing.assert_allclose(hT, rh[0, 0], rtol=0, atol=1e-12 * np.abs(rh).max())


def test_the_walk_needs_the_erase_term():
    """Keys 2 e_1 with beta = 1 on every token: each token multiplies the e_1 row of a
    dropped state by -3 alpha.  The walk with the erase term finds no warm-up within
    4 S tiles, so the sequence runs as one segment and matches the oracle.  A walk
    on the decay alone picks short warm-ups, and its outputs are visibly wrong."""
    rng = np.random.default_rng(301)
    L, dk, dv = 16 * 48, 4, 3
    q = rng.standard_normal((L, dk))
    k = np.zeros((L, dk))
    k[:, 0] = 2.0
    v = rng.standard_normal((L, dv))
    a = np.full((L, dk), -1.0)                    # alpha = e^{-2 sigmoid(-1)} = 0.58 per token
    beta = np.ones(L)
    h0 = rng.standard_normal((dk, dv))
    ro, _ = oracle.oracle_fwd_vec(*(x[None, :, None] for x in (q, k, v, a, beta)), h0=h0[None, None],
                                  b=2.0)
    ro = ro[0, :, 0]
    out, _, warm = _segmented(q, k, v, a, beta, h0, S=4)
    assert warm == {}                               # one segment
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12 * np.abs(ro).max())
    bad, _, warm_bad = _segmented(q, k, v, a, beta, h0, S=4, erase_term=False)
    assert warm_bad and max(s0 - w for s0, w in warm_bad.items()) < 8
    assert np.abs(bad - ro).max() > 1e-3 * np.abs(ro).max()


# ---- the chunked backward's two-sided segments, in fp64 ----------------------------------
def _segmented_bwd(q, k, v, a, beta, h0, dout, dhT, S, b=2.0, horizon=-46.0, chunk=16):
    """One unit, per-channel gate.  The forward chain of each segment starts from a
    zero state at a warm-up tile before it (the sequence start: h0); the adjoint chain
    of each segment starts from a zero gradient at a warm-up tile after its end (the
    sequence end: dhT).  Both warm-ups use the same per-tile bound, sum over the tokens
    of max_d g + ln max(1, |1 - beta |k|^2|) (the adjoint transition is the transpose).
    If a boundary has no warm-up within 4 S tiles on either side, one segment.  Every
    tile's gradients then come from its stored entering state and end gradient.
    Returns (dict of the unit's gradients, number of segments)."""
    L, dk = k.shape
    g = chunk_ref.gate(a, b)
    n_t = (L + chunk - 1) // chunk
    tl = [(c * chunk, min(L, (c + 1) * chunk)) for c in range(n_t)]
    lam = np.array([g[s:e].max(axis=1).sum()
                    + np.log(np.maximum(1.0, np.abs(1.0 - beta[s:e] * (k[s:e] ** 2).sum(1)))).sum()
                    for s, e in tl])
    starts = list(range(0, n_t, S))
    ends = starts[1:] + [n_t]
    fw, aw = {0: 0}, {n_t: n_t}
    for s1 in starts[1:]:
        acc, w = 0.0, None                       # forward chain of the segment starting at s1
        for c in range(s1 - 1, max(-1, s1 - 4 * S - 1), -1):
            acc += lam[c]
            if acc <= horizon:
                w = c
                break
        acc, e = 0.0, None                       # adjoint chain of the segment ending at s1
        for c in range(s1, min(n_t, s1 + 4 * S)):
            acc += lam[c]
            if acc <= horizon:
                e = c + 1
                break
        if (w is None and s1 > 4 * S) or (e is None and s1 + 4 * S < n_t):
            starts, ends, fw, aw = [0], [n_t], {0: 0}, {n_t: n_t}
            break
        fw[s1] = 0 if w is None else w
        aw[s1] = n_t if e is None else e
    H0s, tiles = {}, {}
    for s0, s1 in zip(starts, ends):             # forward chains: entering states of their tiles
        w = fw[s0]
        H = h0.copy() if w == 0 else np.zeros_like(h0)
        for c in range(w, s1):
            s, e = tl[c]
            t = chunk_ref._tile_channels(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], H)
            if c >= s0:
                H0s[c], tiles[c] = H, t
            H = t["H1"]
    res = {n: np.zeros_like(x) for n, x in (("dq", k), ("dk", k), ("dv", v), ("da", a),
                                            ("dbeta", beta))}
    dh0 = None
    for s0, s1 in zip(starts, ends):             # adjoint chains: end gradients, then tile gradients
        e_w = aw[s1]
        dH = dhT.copy() if e_w == n_t else np.zeros_like(dhT)
        for c in range(e_w - 1, s0 - 1, -1):
            s, e = tl[c]
            gq, gk, gv, gg, gb, dH0 = chunk_ref.tile_grads(tiles[c], v[s:e], beta[s:e], dout[s:e], dH)
            if c < s1:
                res["dq"][s:e], res["dk"][s:e], res["dv"][s:e], res["dbeta"][s:e] = gq, gk, gv, gb
                res["da"][s:e] = gg * chunk_ref.gate_grad(a[s:e], b)
            dH = dH0
        if s0 == 0:
            dh0 = dH
    res["dh0"] = dh0
    return res, len(starts)


def test_backward_segments_from_two_sided_warm_ups_reproduce_the_gradients():
    """Unit keys, a ~ N(0, 1), 6 segments of 8 tiles: both chains of every interior
    boundary find warm-ups, and the gradients equal the unsegmented oracle's to
    fp64 rounding."""
    rng = np.random.default_rng(500)
    L, dk, dv = 16 * 48, 8, 6
    q, k, v, _, beta, h0 = _case(rng, L, dk=dk, dv=dv, h0_std=1.0)
    a = rng.standard_normal((1, L, 1, dk))
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    got, nseg = _segmented_bwd(q[0, :, 0], k[0, :, 0], v[0, :, 0], a[0, :, 0], beta[0, :, 0],
                               h0[0, 0], dout[0, :, 0], dhT[0, 0], S=8)
    assert nseg == 6
    ref = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    for n in ("dq", "dk", "dv", "da", "dbeta"):
        r = ref[n][0, :, 0]
        np.testing.assert_allclose(got[n], r, rtol=0, atol=1e-11 * max(1.0, np.abs(r).max()), err_msg=n)
    np.testing.assert_allclose(got["dh0"], ref["dh0"][0, 0], rtol=0,
                               atol=1e-11 * max(1.0, np.abs(ref["dh0"]).max()))


def test_backward_segments_with_a_short_horizon_are_visible():
    """Where the bound is tight, a short horizon shows.  Every channel shares one gate
    (a ~ N(-2, 1)) and beta = 1e-3, so a dropped state or gradient shrinks almost
    exactly by the bound.  With the horizon at -46 the segmented gradients equal the
    oracle's to rounding.  At -3 the dropped parts (about e^-3) show in dk and dv."""
    rng = np.random.default_rng(501)
    L, dk, dv = 16 * 48, 8, 6
    q, k, v, _, beta, h0 = _case(rng, L, dk=dk, dv=dv, h0_std=1.0)
    a = np.repeat((rng.standard_normal((1, L, 1)) - 2.0)[..., None], dk, axis=-1)
    beta = np.full(beta.shape, 1e-3)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    ref = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    args = (q[0, :, 0], k[0, :, 0], v[0, :, 0], a[0, :, 0], beta[0, :, 0], h0[0, 0], dout[0, :, 0],
            dhT[0, 0])
    exact, nseg = _segmented_bwd(*args, S=8)
    short, nseg_s = _segmented_bwd(*args, S=8, horizon=-3.0)
    assert nseg == nseg_s == 6
    for n in ("dk", "dv"):
        scale = np.abs(ref[n]).max()
        assert np.abs(exact[n] - ref[n][0, :, 0]).max() <= 1e-12 * scale
        assert np.abs(short[n] - ref[n][0, :, 0]).max() > 1e-3 * scale
