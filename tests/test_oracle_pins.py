"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: values printed on the pages (tests/golden), closed forms, brute-force
dense matrix products on tiny inputs, identities and a norm bound.  Together
they are chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them.

Citation keys (page title, section):
  P1 = "Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs"
  P2 = "Core Technologies Behind Ultra-Long-Context Sparse MoE Large Models"
  P3 = "How Trillion-Scale Sparse MoE Models Achieve Million-Token Long Context
        Capabilities"
  P4 = "Evaluating Next-Gen Sparse MoE and Long-Context LLMs"
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunk_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gate_bounds.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv, src = line.split(";", 1)
            key, val = (s.strip() for s in kv.split("="))
            assert src.strip(), f"{key} has no citation"
            vals[key] = float(val)
    return vals


def _rand_unit(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _case(rng, T, H=1, dk=8, dv=6, B=1, a_std=1.0, h0_std=0.3):
    q = _rand_unit(rng, B * T * H, dk).reshape(B, T, H, dk)
    k = _rand_unit(rng, B * T * H, dk).reshape(B, T, H, dk)
    v = rng.standard_normal((B, T, H, dv))
    a = a_std * rng.standard_normal((B, T, H))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = h0_std * rng.standard_normal((B, H, dk, dv))
    return q, k, v, a, beta, h0


def _g(a, b=2.0, mode="bounded"):
    return np.vectorize(lambda x: oracle.gate(x, b, mode))(a)


# --------------------------------------------------------------------------
# gate: the pages' printed range [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3]
# --------------------------------------------------------------------------
def test_gate_range_matches_pages():
    gv = _golden()
    bnd = -gv["g_min"]                   # g = g_min * sigmoid(x), g_min = -5
    a = np.linspace(-60, 60, 2001)
    g = _g(a, bnd)
    assert g.min() >= gv["g_min"] - 1e-12 and g.max() <= gv["g_max"]
    assert abs(oracle.gate(60.0, bnd) - gv["g_min"]) < 1e-12
    assert abs(oracle.gate(-60.0, bnd)) < 1e-20
    decay = np.exp(g)
    # exp(g) in approximately [0.0067, 1]
    assert abs(decay.min() - gv["decay_min_approx"]) < 5e-5
    assert decay.max() <= gv["decay_max"]
    # exp(-g) in [1, e^5 ~ 148]
    recip = np.exp(-g)
    assert recip.min() >= gv["recip_min"] - 1e-15
    assert abs(recip.max() - gv["recip_max_approx"]) < 0.5


def test_gate_tile_reciprocal_fits_bf16_only_when_bounded():
    """Within a 16-token tile the reciprocal of the cumulative decay stays
    inside bf16's range under the bounded gate, and can leave it under the
    unbounded softplus gate [P2 §2.1-2.2, P3 §3.1-3.2, P4 §2.3]."""
    gv = _golden()
    tile = int(gv["tile"])
    bf16_max = float(torch.finfo(torch.bfloat16).max)
    worst_bounded = math.exp(-tile * oracle.gate(80.0, -gv["g_min"]))
    assert worst_bounded < bf16_max
    worst_softplus = -tile * oracle.gate(10.0, 0.0, "softplus")   # ~ 160
    assert worst_softplus > math.log(bf16_max)


@pytest.mark.parametrize("C,b,overflows", [(16, 2.0, False), (16, 8.0, True), (32, 2.0, False),
                                             (32, 8.0, True), (64, 2.0, False), (64, 8.0, True)])
def test_factored_tile_form_breaks_where_the_tile_decay_leaves_fp32(C, b, overflows):
    """Where the factored in-tile form (Q (.) e^G)(K (.) e^-G)^T breaks, on the gate
    recipe of the 32-head, 65,536-token workload (a ~ N(0, 2)).  The form needs
    e^{-G} inside fp32, i.e. an in-tile |G| below ln(FLT_MAX) = 88.7.  Over 65,536
    tokens the largest in-tile |G| stays below that for b = 2 at C = 16, 32 and 64
    (at most b C = 32, 64, 128; 78.8 reached at C = 64).  It exceeds that for b = 8 at
    every C.  In the worst tile the factored fp32 Gram then has non-finite entries on
    and below the diagonal, while the pairwise form (e^{G_i - G_j} <= 1, the one the
    scalar kernels use) stays finite for every case."""
    rng = np.random.default_rng(1002)
    a = 2.0 * rng.standard_normal(65536)
    g = -b / (1.0 + np.exp(-a))                     # the bounded gate, restated in numpy
    np.testing.assert_allclose(g[:64], _g(a[:64], b), rtol=1e-15, atol=0)
    n = len(g) // C
    G = np.cumsum(g[: n * C].reshape(n, C), axis=1)
    worst = int(np.argmin(G[:, -1]))
    f32_max_log = math.log(float(np.finfo(np.float32).max))
    assert (-G[worst, -1] > f32_max_log) == overflows
    Gt = G[worst].astype(np.float32)
    q = _rand_unit(rng, C, 16).astype(np.float32)
    k = _rand_unit(rng, C, 16).astype(np.float32)
    lower = np.tril(np.ones((C, C), dtype=bool))
    with np.errstate(over="ignore", invalid="ignore"):
        factored = (q * np.exp(Gt)[:, None]) @ (k * np.exp(-Gt)[:, None]).T
    pairwise = (q @ k.T) * np.exp(np.where(lower, Gt[:, None] - Gt[None, :], np.float32(-np.inf)))
    assert np.isfinite(pairwise).all()
    assert bool(np.isfinite(factored[lower]).all()) == (not overflows)


def test_gate_symmetry_and_softplus():
    rng = np.random.default_rng(1)
    for b in (2.0, 5.0, 8.0):
        for a in rng.standard_normal(50) * 4:
            # sigmoid(-a) = 1 - sigmoid(a)  =>  g(-a) = -b - g(a)
            assert abs(oracle.gate(-a, b) + b + oracle.gate(a, b)) < 1e-12
            assert abs(oracle.gate(a, b) - (-b / (1 + math.exp(-a)))) < 1e-12
    for a in (-30.0, -3.0, 0.0, 0.5, 3.0, 30.0, 700.0):
        ref = -(a + math.log1p(math.exp(-a))) if a > 0 else -math.log1p(math.exp(a))
        assert abs(oracle.gate(a, 0.0, "softplus") - ref) <= 1e-12 * max(1.0, abs(a))
    assert abs(oracle.gate(0.0, 0.0, "softplus") + math.log(2.0)) < 1e-15


# --------------------------------------------------------------------------
# recurrence: brute-force unrolled dense products (T <= 32)
# --------------------------------------------------------------------------
def _brute_force(q, k, v, g, beta, h0):
    """H_t = Phi_t H_{t-1} + beta_t k_t v_t^T with Phi_t = alpha_t (I - beta_t k_t k_t^T),
    expanded as H_t = Phi_{1:t} h0 + sum_s Phi_{s+1:t} beta_s k_s v_s^T, with
    every Phi a dense dk x dk matrix; o_t = H_t^T q_t."""
    T, dk = k.shape
    Phi = [math.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    out = np.zeros((T, v.shape[1]))
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


@pytest.mark.parametrize("T,dk,dv,b,mode", [(1, 4, 3, 2.0, "bounded"),
                                             (7, 8, 5, 2.0, "bounded"),
                                             (32, 8, 6, 8.0, "bounded"),
                                             (20, 6, 6, 0.0, "softplus")])
def test_recurrence_matches_unrolled_products(T, dk, dv, b, mode):
    rng = np.random.default_rng(T * 100 + dk)
    q, k, v, a, beta, h0 = _case(rng, T, dk=dk, dv=dv)
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=b, gate=mode)
    g = chunk_ref.gate(a[0, :, 0], b, mode)
    ref_o, ref_h = _brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    np.testing.assert_allclose(out[0, :, 0], ref_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], ref_h, rtol=1e-11, atol=1e-12)


def test_unnormalised_keys_and_wide_beta():
    """The brute-force pin also holds away from the unit-norm / beta in [0,1]
    regime, so no normalisation is hidden in the oracle."""
    rng = np.random.default_rng(7)
    q, k, v, a, beta, h0 = _case(rng, 9, dk=5, dv=4)
    k = k * 1.7
    beta = beta * 1.5
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=3.0)
    g = chunk_ref.gate(a[0, :, 0], 3.0)
    ref_o, ref_h = _brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    np.testing.assert_allclose(out[0, :, 0], ref_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], ref_h, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_beta_zero_is_pure_decay():
    """beta = 0 writes nothing: o_t = exp(sum_{r<=t} g_r) h0^T q_t, hT = exp(sum g) h0."""
    rng = np.random.default_rng(3)
    q, k, v, a, beta, h0 = _case(rng, 40, H=2, dk=8, dv=8, B=2)
    beta[:] = 0.0
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    for n in range(2):
        for h in range(2):
            cg = np.cumsum(chunk_ref.gate(a[n, :, h], 2.0))
            ref = np.exp(cg)[:, None] * (q[n, :, h] @ h0[n, h])
            np.testing.assert_allclose(out[n, :, h], ref, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(hT[n, h], math.exp(cg[-1]) * h0[n, h], rtol=1e-12)


def _gla_closed_form(q, k, v, g, beta, h0):
    T = q.shape[0]
    cg = np.concatenate([[0.0], np.cumsum(g)])
    out = np.zeros((T, v.shape[1]))
    for t in range(T):
        acc = math.exp(cg[t + 1]) * (h0.T @ q[t])
        for s in range(t + 1):
            acc = acc + math.exp(cg[t + 1] - cg[s + 1]) * beta[s] * (q[t] @ k[s]) * v[s]
        out[t] = acc
    return out


def test_no_erase_is_gated_linear_attention():
    """Without the erase term the recurrence is gated linear attention:
    o_t = sum_{s<=t} exp(sum_{s<r<=t} g_r) beta_s (q_t.k_s) v_s (+ decayed h0)."""
    rng = np.random.default_rng(4)
    q, k, v, a, beta, h0 = _case(rng, 30, dk=8, dv=5)
    out, _ = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0, erase=False)
    g = chunk_ref.gate(a[0, :, 0], 2.0)
    ref = _gla_closed_form(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    np.testing.assert_allclose(out[0, :, 0], ref, rtol=1e-11, atol=1e-13)


def test_orthogonal_keys_reduce_to_gla():
    """Mutually orthogonal unit keys (T <= dk) make the erase term vanish, so
    the delta rule equals the gated linear-attention closed form."""
    rng = np.random.default_rng(5)
    T, dk, dv = 16, 16, 7
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    q, k, v, a, beta, _ = _case(rng, T, dk=dk, dv=dv)
    k[0, :, 0] = Qm[:, :T].T
    out, _ = oracle.oracle_fwd(q, k, v, a, beta, b=2.0)
    g = chunk_ref.gate(a[0, :, 0], 2.0)
    ref = _gla_closed_form(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], np.zeros((dk, dv)))
    np.testing.assert_allclose(out[0, :, 0], ref, rtol=1e-11, atol=1e-13)


def test_overwrite_identity():
    """g = 0, beta = 1, unit keys: the delta rule stores v_t under k_t exactly,
    H_t^T k_t = v_t for every t and any keys; with orthonormal keys every earlier
    association persists, H_T^T k_s = v_s."""
    rng = np.random.default_rng(6)
    T, dk, dv = 12, 12, 5
    q, k, v, _, _, h0 = _case(rng, T, dk=dk, dv=dv)
    beta = np.ones((1, T, 1))
    a = np.full((1, T, 1), -800.0)          # sigmoid(-800) = 0 exactly -> g = 0
    # q_t = k_t makes o_t = H_t^T k_t
    qq = q.copy()
    qq[0, :, 0] = k[0, :, 0]
    out, _ = oracle.oracle_fwd(qq, k, v, a, beta, h0=h0, b=2.0)
    np.testing.assert_allclose(out[0, :, 0], v[0, :, 0], rtol=1e-12, atol=1e-12)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k[0, :, 0] = Qm.T
    _, hT = oracle.oracle_fwd(q, k, v, a, beta, b=2.0)
    np.testing.assert_allclose(k[0, :, 0] @ hT[0, 0], v[0, :, 0], rtol=1e-12, atol=1e-12)


def test_state_norm_bound_along_trajectory():
    """||H_t||_2 <= alpha_t ||H_{t-1}||_2 + beta_t ||v_t|| ||k_t|| for unit k and
    beta in [0,1], because ||I - beta k k^T||_2 = 1.  The trajectory is taken
    one token at a time by chaining hT into h0."""
    rng = np.random.default_rng(8)
    q, k, v, a, beta, h0 = _case(rng, 48, dk=8, dv=8, h0_std=1.0)
    H = h0.copy()
    for t in range(48):
        sl = slice(t, t + 1)
        _, Hn = oracle.oracle_fwd(q[:, sl], k[:, sl], v[:, sl], a[:, sl], beta[:, sl], h0=H, b=2.0)
        alpha = math.exp(oracle.gate(a[0, t, 0], 2.0))
        bound = alpha * np.linalg.norm(H[0, 0], 2) + beta[0, t, 0] * np.linalg.norm(v[0, t, 0]) \
            * np.linalg.norm(k[0, t, 0])
        assert np.linalg.norm(Hn[0, 0], 2) <= bound * (1 + 1e-12)
        H = Hn


def test_dropped_state_decays_with_the_gate_for_unit_keys():
    """The tensor-core path's segment truncation: for unit keys and beta in [0, 1] the
    erase factors have norm <= 1, so two runs over the same tokens from different
    entering states stay within prod_t alpha_t of their entering difference.
    Outside that precondition (beta |k|^2 = 3, an erase factor of norm 2) the
    decay-only product is exceeded."""
    rng = np.random.default_rng(9)
    T, dk, dv = 12, 8, 6   # the product of decays stays far above fp64 rounding of the states
    q, k, v, a, beta, h0 = _case(rng, T, dk=dk, dv=dv, h0_std=1.0)
    h1 = rng.standard_normal(h0.shape)
    _, Ha = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    _, Hb = oracle.oracle_fwd(q, k, v, a, beta, h0=h1, b=2.0)
    decay = math.exp(sum(oracle.gate(x, 2.0) for x in a[0, :, 0]))
    assert decay > 1e-8
    slack = 1e-14 * max(np.linalg.norm(Ha), np.linalg.norm(Hb))
    assert np.linalg.norm(Hb - Ha) <= decay * np.linalg.norm(h1 - h0) * (1 + 1e-9) + slack
    # every key e_1 scaled to |k|^2 = 3, beta = 1: the e_1 row is multiplied by -2 alpha
    k3 = np.zeros_like(k)
    k3[..., 0] = math.sqrt(3.0)
    ones = np.ones_like(beta)
    a8 = np.full_like(a, -8.0)
    d = np.zeros_like(h0)
    d[0, 0, 0] = rng.standard_normal(dv)
    _, Ha = oracle.oracle_fwd(q, k3, v, a8, ones, h0=h0, b=2.0)
    _, Hb = oracle.oracle_fwd(q, k3, v, a8, ones, h0=h0 + d, b=2.0)
    alpha = math.exp(oracle.gate(-8.0, 2.0))
    np.testing.assert_allclose(np.linalg.norm(Hb - Ha), (2 * alpha) ** T * np.linalg.norm(d), rtol=1e-9)
    assert np.linalg.norm(Hb - Ha) > 1e3 * alpha ** T * np.linalg.norm(d)   # 2^12 = 4096


def test_chaining_and_varlen_equal_separate_calls():
    """fwd(x[0:T]) == fwd(x[s:T], h0 = fwd(x[0:s]).hT), and a packed varlen call
    equals one call per sequence."""
    rng = np.random.default_rng(9)
    q, k, v, a, beta, h0 = _case(rng, 50, H=3, dk=8, dv=4)
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0)
    s = 17
    o1, h1 = oracle.oracle_fwd(q[:, :s], k[:, :s], v[:, :s], a[:, :s], beta[:, :s], h0=h0)
    o2, h2 = oracle.oracle_fwd(q[:, s:], k[:, s:], v[:, s:], a[:, s:], beta[:, s:], h0=h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), out, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, hT, rtol=1e-13, atol=1e-14)
    cu = np.array([0, 5, 5, 23, 50])
    h0v = rng.standard_normal((4, 3, 8, 4))
    ov, hv = oracle.oracle_fwd(q, k, v, a, beta, h0=h0v, cu_seqlens=cu)
    for n in range(4):
        sl = slice(cu[n], cu[n + 1])
        on, hn = oracle.oracle_fwd(q[:, sl], k[:, sl], v[:, sl], a[:, sl], beta[:, sl], h0=h0v[n:n + 1])
        np.testing.assert_allclose(ov[:, sl], on, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hv[n], hn[0], rtol=1e-13, atol=1e-14)


def test_bf16_inputs_are_widened_exactly():
    rng = np.random.default_rng(10)
    q, k, v, a, beta, h0 = _case(rng, 20, H=2, dk=8, dv=8)
    t = [torch.from_numpy(x).to(torch.bfloat16) for x in (q, k, v, a, beta)]
    o_bf, h_bf = oracle.oracle_fwd(*t, h0=h0)
    o_64, h_64 = oracle.oracle_fwd(*[x.double().numpy() for x in t], h0=h0)
    np.testing.assert_array_equal(o_bf, o_64)
    np.testing.assert_array_equal(h_bf, h_64)


# --------------------------------------------------------------------------
# the chunked (WY / UT) form is the same function
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T,chunk", [(32, 32), (16, 16), (50, 16), (64, 32), (70, 64)])
def test_chunk_form_equals_token_oracle(T, chunk):
    rng = np.random.default_rng(T + chunk)
    q, k, v, a, beta, h0 = _case(rng, T, H=2, dk=8, dv=6)
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0)
    oc, hc = chunk_ref.fwd(q, k, v, a, beta, h0=h0, chunk=chunk, b=2.0)
    np.testing.assert_allclose(oc, out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hc, hT, rtol=1e-10, atol=1e-12)


def test_chunk_form_softplus_and_varlen():
    rng = np.random.default_rng(11)
    q, k, v, a, beta, _ = _case(rng, 45, H=2, dk=8, dv=6, a_std=3.0)
    cu = np.array([0, 13, 14, 45])
    h0 = rng.standard_normal((3, 2, 8, 6)) * 0.1
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, cu_seqlens=cu, gate="softplus")
    oc, hc = chunk_ref.fwd(q, k, v, a, beta, h0=h0, cu_seqlens=cu, chunk=16, mode="softplus")
    np.testing.assert_allclose(oc, out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hc, hT, rtol=1e-10, atol=1e-12)


def test_tile_inverse_against_dense_solve():
    """T = (I + A)^{-1} from the triangular solver agrees with a dense general
    inverse, and A is strictly lower triangular with the decay-scaled Gram."""
    rng = np.random.default_rng(12)
    C, dk = 16, 8
    k = _rand_unit(rng, C, dk)
    v = rng.standard_normal((C, 4))
    beta = rng.uniform(0, 1, C)
    G = np.cumsum(chunk_ref.gate(rng.standard_normal(C), 2.0))
    A, T, W, U = chunk_ref.tile_wy(k, v, beta, G)
    assert np.all(np.triu(A) == 0)
    i, j = 9, 4
    assert abs(A[i, j] - beta[i] * math.exp(G[i] - G[j]) * (k[i] @ k[j])) < 1e-15
    np.testing.assert_allclose(T, np.linalg.inv(np.eye(C) + A), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose((np.eye(C) + A) @ U, beta[:, None] * v, rtol=1e-12, atol=1e-12)
