"""Pins of the per-channel decay oracle (``oracle_fwd_vec``), CPU only.

The per-channel form gives every key channel i its own decay factor
alpha_{t,i} = exp(g(a_{t,i})) and applies it to row i of the dk x dv state
before the delta-rule write:  H_t = (I - beta_t k_t k_t^T) diag(alpha_t) H_{t-1}
+ beta_t k_t v_t^T,  o_t = H_t^T q_t.  The pins check it against:
  - the scalar oracle (itself pinned elsewhere) when all channels share a;
  - a brute-force expansion in dense dk x dk transition matrices;
  - the closed form of per-channel gated linear attention when the erase term
    is dropped;
  - beta = 0 (pure per-channel decay) and one-hot keys (only that row is
    rewritten, every other row only decays).
Its backward (``oracle_bwd_vec``) is pinned by finite differences of the forward
and by its reduction to the scalar backward when all channels share a.
The bound that places the segmented kernels' warm-up tiles is checked on the
oracle's trajectories: the norm identity of the erase factor, the per-token maximum
decay, and that the bound's product dominates the effect of a dropped entering
state (and that its erase-factor term cannot be left out).
Planted one-token mistakes in copies of the C source must fail the battery.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from test_oracle_pins import _case, _g

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")


def _vec_case(rng, T, H=1, dk=6, dv=5, B=1, a_std=1.0):
    q, k, v, _, beta, h0 = _case(rng, T, H=H, dk=dk, dv=dv, B=B)
    a = a_std * rng.standard_normal((B, T, H, dk))
    return q, k, v, a, beta, h0


def _brute_force_vec(q, k, v, g, beta, h0):
    """Dense transitions Phi_t = (I - beta k k^T) diag(exp(g_t)); H_t expanded as
    Phi_{1:t} h0 + sum_s Phi_{s+1:t} beta_s k_s v_s^T."""
    T, dk = k.shape
    Phi = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t])) for t in range(T)]
    out = np.zeros((T, v.shape[1]))
    Ht = h0
    for t in range(T):
        P = np.eye(dk)
        for r in range(t, -1, -1):
            P = P @ Phi[r]
        Ht = P @ h0
        for s in range(t + 1):
            Ps = np.eye(dk)
            for r in range(t, s, -1):
                Ps = Ps @ Phi[r]
            Ht = Ht + Ps @ (beta[s] * np.outer(k[s], v[s]))
        out[t] = Ht.T @ q[t]
    return out, Ht


def test_equal_channels_reduce_to_scalar_oracle():
    rng = np.random.default_rng(21)
    q, k, v, _, beta, h0 = _case(rng, 50, H=2, dk=8, dv=6, B=2)
    a = rng.standard_normal((2, 50, 2))
    av = np.repeat(a[..., None], 8, axis=-1)
    for gate, b in (("bounded", 2.0), ("softplus", 0.0)):
        o1, h1 = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=b, gate=gate)
        o2, h2 = oracle.oracle_fwd_vec(q, k, v, av, beta, h0=h0, b=b, gate=gate)
        np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h2, h1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T,dk,dv,b", [(1, 4, 3, 2.0), (9, 6, 5, 2.0), (24, 8, 4, 5.0)])
def test_matches_dense_transition_products(T, dk, dv, b):
    rng = np.random.default_rng(30 + T)
    q, k, v, a, beta, h0 = _vec_case(rng, T, dk=dk, dv=dv)
    out, hT = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=b)
    g = _g(a[0, :, 0], b)
    ro, rh = _brute_force_vec(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    np.testing.assert_allclose(out[0, :, 0], ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], rh, rtol=1e-11, atol=1e-12)


def test_no_erase_is_per_channel_gated_linear_attention():
    """Without the erase term: o_t = sum_{s<=t} beta_s sum_i q_ti k_si
    exp(G_ti - G_si) v_s + sum_i q_ti exp(G_ti) h0[i], G the per-channel cumsum."""
    rng = np.random.default_rng(22)
    T, dk, dv = 20, 6, 4
    q, k, v, a, beta, h0 = _vec_case(rng, T, dk=dk, dv=dv)
    out, _ = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=2.0, erase=False)
    G = np.cumsum(_g(a[0, :, 0], 2.0), axis=0)
    qq, kk, vv, bb = q[0, :, 0], k[0, :, 0], v[0, :, 0], beta[0, :, 0]
    ref = np.zeros((T, dv))
    for t in range(T):
        acc = (qq[t] * np.exp(G[t])) @ h0[0, 0]
        for s in range(t + 1):
            acc = acc + bb[s] * float(np.sum(qq[t] * kk[s] * np.exp(G[t] - G[s]))) * vv[s]
        ref[t] = acc
    np.testing.assert_allclose(out[0, :, 0], ref, rtol=1e-11, atol=1e-13)


def test_beta_zero_is_per_channel_decay():
    rng = np.random.default_rng(23)
    q, k, v, a, beta, h0 = _vec_case(rng, 30, H=2, dk=5, dv=4, B=2)
    beta[:] = 0.0
    out, hT = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=2.0)
    for n in range(2):
        for h in range(2):
            G = np.cumsum(_g(a[n, :, h], 2.0), axis=0)       # [T, dk]
            ref = np.stack([(q[n, t, h] * np.exp(G[t])) @ h0[n, h] for t in range(30)])
            np.testing.assert_allclose(out[n, :, h], ref, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(hT[n, h], np.exp(G[-1])[:, None] * h0[n, h], rtol=1e-12)


def test_one_hot_key_rewrites_only_its_row():
    """k = e_r, beta = 1: row r of H becomes v_t, every other row i only decays
    by exp(g_{t,i})."""
    rng = np.random.default_rng(24)
    T, dk, dv = 6, 5, 3
    q, k, v, a, beta, h0 = _vec_case(rng, T, dk=dk, dv=dv)
    beta[:] = 1.0
    rows = [2, 0, 4, 2, 1, 3]
    k[:] = 0.0
    for t, r in enumerate(rows):
        k[0, t, 0, r] = 1.0
    _, hT = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=2.0)
    g = _g(a[0, :, 0], 2.0)
    H = h0[0, 0].copy()
    for t, r in enumerate(rows):
        H = np.exp(g[t])[:, None] * H
        H[r] = v[0, t, 0]
    np.testing.assert_allclose(hT[0, 0], H, rtol=1e-13, atol=1e-15)


# one-token edits of the per-channel forward in gdr_oracle.c
VEC_MUTANTS = {
    "decay_after_prediction": ("Hs[i * CB + c] *= al[i];\n                        p += kt[i] * Hs[i * CB + c];",
                               "p += kt[i] * Hs[i * CB + c];\n                        Hs[i * CB + c] *= al[i];"),
    "one_factor_for_all_rows": ("Hs[i * CB + c] *= al[i];", "Hs[i * CB + c] *= al[0];"),
    "gate_reads_channel_zero": ("widen(a, in_dtype, row * dk + i)", "widen(a, in_dtype, row * dk)"),
    "erase_dropped": ("(erase ? p : 0.0)", "0.0"),
}


@pytest.mark.parametrize("name", list(VEC_MUTANTS))
def test_vec_mutant_is_rejected(tmp_path, name):
    old, new = VEC_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    c, so = tmp_path / f"{name}.c", tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(c),
                    "-lm"], check=True)
    rng = np.random.default_rng(31)
    q, k, v, a, beta, h0 = _vec_case(rng, 9, dk=6, dv=5)
    out, hT = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=2.0, _lib_path=str(so))
    g = _g(a[0, :, 0], 2.0)
    ro, rh = _brute_force_vec(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    ok = np.allclose(out[0, :, 0], ro, rtol=1e-11, atol=1e-12) and \
        np.allclose(hT[0, 0], rh, rtol=1e-11, atol=1e-12)
    assert not ok


# --------------------------------------------------------------------------
# per-channel backward (oracle_bwd_vec)
# --------------------------------------------------------------------------
def _vec_loss(x, dout, dhT, b, cu=None):
    out, hT = oracle.oracle_fwd_vec(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"],
                                    cu_seqlens=cu, b=b)
    return float((out * dout).sum() + (hT * dhT).sum())


@pytest.mark.parametrize("T,dk,dv,varlen", [(6, 3, 4, False), (40, 4, 3, False), (30, 3, 2, True)])
def test_vec_backward_matches_finite_differences(T, dk, dv, varlen):
    rng = np.random.default_rng(40 + T)
    q, k, v, a, beta, h0 = _vec_case(rng, T, H=2, dk=dk, dv=dv)
    cu = np.array([0, 4, 4, T], dtype=np.int64) if varlen else None
    N = 3 if varlen else 1
    h0 = 0.3 * rng.standard_normal((N, 2, dk, dv))
    x = dict(q=q, k=k, v=v, a=a, beta=beta, h0=h0)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal((N, 2, dk, dv))
    g = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, cu_seqlens=cu, b=2.0)
    grads = {"q": g["dq"], "k": g["dk"], "v": g["dv"], "a": g["da"], "beta": g["dbeta"],
             "h0": g["dh0"]}
    eps = 1e-5
    for name, grad in grads.items():
        R = rng.standard_normal(x[name].shape)
        fd = (_vec_loss(dict(x, **{name: x[name] + eps * R}), dout, dhT, 2.0, cu)
              - _vec_loss(dict(x, **{name: x[name] - eps * R}), dout, dhT, 2.0, cu)) / (2 * eps)
        an = float((grad * R).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_vec_backward_with_equal_channels_is_the_scalar_backward():
    """All channels sharing a: every gradient equals the scalar backward's, and the
    per-channel da summed over the channels equals the scalar da."""
    rng = np.random.default_rng(41)
    q, k, v, _, beta, h0 = _case(rng, 25, H=2, dk=5, dv=4, B=2)
    a = rng.standard_normal((2, 25, 2))
    av = np.repeat(a[..., None], 5, axis=-1)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    gs = oracle.oracle_bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    gv = oracle.oracle_bwd_vec(q, k, v, av, beta, dout=dout, dhT=dhT, h0=h0, b=2.0)
    for name in ("dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(gv[name], gs[name], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(gv["da"].sum(axis=-1), gs["da"], rtol=1e-11, atol=1e-12)


VEC_BWD_MUTANTS = {
    "k_grad_without_row_decay": ("gk += dH[i * dv + j] * de[j] + al[i] * Hp[i * dv + j] * gp[j];",
                                 "gk += dH[i * dv + j] * de[j] + Hp[i * dv + j] * gp[j];"),
    "decay_grad_reads_new_state": ("dal += Hp[i * dv + j] * hb_bar;", "dal += Ht[i * dv + j] * hb_bar;"),
}


@pytest.mark.parametrize("name", list(VEC_BWD_MUTANTS))
def test_vec_backward_mutant_is_rejected(tmp_path, name):
    old, new = VEC_BWD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    c, so = tmp_path / f"{name}.c", tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(c),
                    "-lm"], check=True)
    rng = np.random.default_rng(42)
    q, k, v, a, beta, h0 = _vec_case(rng, 8, dk=4, dv=3)
    x = dict(q=q, k=k, v=v, a=a, beta=beta, h0=h0)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    g = oracle.oracle_bwd_vec(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, b=2.0, _lib_path=str(so))
    grads = {"q": g["dq"], "k": g["dk"], "v": g["dv"], "a": g["da"], "beta": g["dbeta"],
             "h0": g["dh0"]}
    caught = False
    for xname, grad in grads.items():
        R = rng.standard_normal(x[xname].shape)
        fd = (_vec_loss(dict(x, **{xname: x[xname] + 1e-5 * R}), dout, dhT, 2.0)
              - _vec_loss(dict(x, **{xname: x[xname] - 1e-5 * R}), dout, dhT, 2.0)) / 2e-5
        caught |= abs(fd - float((grad * R).sum())) > 1e-6 * max(1.0, abs(fd))
    assert caught


# --------------------------------------------------------------------------
# the bound behind the segmented per-channel kernels' warm-up tiles
# --------------------------------------------------------------------------
def test_erase_factor_norm_identity():
    """||I - beta k k^T||_2 = max(1, |1 - beta |k|^2|): its eigenvalues are 1 (dk - 1
    times, on the complement of k) and 1 - beta |k|^2 (on k).  Checked against the
    matrix 2-norm for unit and unnormalised keys and beta outside [0, 1]."""
    rng = np.random.default_rng(41)
    for _ in range(300):
        dk = int(rng.integers(2, 10))
        k = rng.standard_normal(dk) * rng.choice([0.3, 1.0, 2.0])
        beta = rng.uniform(-0.5, 2.0)
        want = max(1.0, abs(1.0 - beta * float(k @ k)))
        got = np.linalg.norm(np.eye(dk) - beta * np.outer(k, k), 2)
        assert abs(got - want) <= 1e-12 * want


def test_channel_decay_maximum_is_the_gate_at_the_smallest_input():
    """max_d exp(g(a_d)) = exp(g(min_d a)) for the bounded gate (g is decreasing in
    a), so the bound needs one minimum per token, not dk exponentials."""
    rng = np.random.default_rng(42)
    for b in (0.5, 2.0, 5.0):
        a = 3.0 * rng.standard_normal((100, 16))
        full = np.exp(_g(a, b)).max(axis=1)
        short = np.exp(_g(a.min(axis=1), b))
        np.testing.assert_array_equal(full, short)


@pytest.mark.parametrize("key_scale,beta_hi", [(1.0, 1.0), (2.0, 1.0), (1.0, 2.0)])
def test_warm_up_bound_dominates_the_dropped_state(key_scale, beta_hi):
    """Two runs over the same tokens from different entering states differ by the
    transitions applied to the difference (the recurrence is affine in the state).
    After every token the difference stays within
        prod_t max(1, |1 - beta_t |k_t|^2|) max_d alpha_{t,d}
    times the entering one: the bound that places the warm-up tiles.  Each run is
    taken one token at a time by chaining hT into h0; unnormalised keys and beta > 1
    make some tokens' erase factors expansive."""
    rng = np.random.default_rng(43)
    T, dk, dv, b = 64, 8, 6, 2.0
    q, k, v, a, beta, h0 = _vec_case(rng, T, dk=dk, dv=dv)
    k = k * key_scale
    beta = rng.uniform(0.0, beta_hi, beta.shape)
    h1 = rng.standard_normal(h0.shape)
    d0 = np.linalg.norm(h1 - h0)
    Ha, Hb = h0.copy(), h1.copy()
    log_bound = 0.0
    for t in range(T):
        sl = slice(t, t + 1)
        _, Ha = oracle.oracle_fwd_vec(q[:, sl], k[:, sl], v[:, sl], a[:, sl], beta[:, sl], h0=Ha, b=b)
        _, Hb = oracle.oracle_fwd_vec(q[:, sl], k[:, sl], v[:, sl], a[:, sl], beta[:, sl], h0=Hb, b=b)
        kt, bt = k[0, t, 0], beta[0, t, 0]
        log_alpha_max = float(_g(a[0, t, 0].min(), b))
        log_bound += log_alpha_max + math.log(max(1.0, abs(1.0 - bt * float(kt @ kt))))
        dt = np.linalg.norm(Hb - Ha)
        assert dt <= math.exp(log_bound) * d0 * (1 + 1e-9), (t, dt, math.exp(log_bound) * d0)


def test_erase_factor_term_is_needed():
    """Every key 2 e_1 with beta = 1 and an almost undamped gate (a = -8): each token
    multiplies the e_1 row of the state difference by 1 - 4 = -3.  The decay-only
    product prod_t max_d alpha_{t,d} (about 1) is exceeded, while the bound with
    the erase factor's term (3 alpha per token) holds, here with equality."""
    T, dk, dv, b = 6, 4, 3, 2.0
    rng = np.random.default_rng(44)
    q = rng.standard_normal((1, T, 1, dk))
    k = np.zeros((1, T, 1, dk))
    k[..., 0] = 2.0
    v = rng.standard_normal((1, T, 1, dv))
    a = np.full((1, T, 1, dk), -8.0)
    beta = np.ones((1, T, 1))
    h0 = np.zeros((1, 1, dk, dv))
    h1 = h0.copy()
    h1[0, 0, 0] = rng.standard_normal(dv)        # the difference lies in the e_1 row
    d0 = np.linalg.norm(h1 - h0)
    _, Ha = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h0, b=b)
    _, Hb = oracle.oracle_fwd_vec(q, k, v, a, beta, h0=h1, b=b)
    dT = np.linalg.norm(Hb - Ha)
    alpha = math.exp(float(_g(-8.0, b)))
    assert dT > 100 * alpha ** T * d0                  # decay-only bound: far exceeded
    np.testing.assert_allclose(dT, (3.0 * alpha) ** T * d0, rtol=1e-12)
