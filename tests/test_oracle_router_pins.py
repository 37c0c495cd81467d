"""Pins of the router-bias oracle (``oracle.router_topk`` / ``router_update``), CPU only.

The oracle follows the quantile-balancing update of "Deep Dive: The Next
Generation of Ultra-Long Context Sparse MoE LLMs" §4.2, "Core Technologies
Behind Ultra-Long-Context Sparse MoE Large Models" §3.2, "How Trillion-Scale
Sparse MoE Models Achieve Million-Token Long Context Capabilities" §4.3 and
"Evaluating Next-Gen Sparse MoE and Long-Context LLMs" §3.2.  Its pieces are
pinned to library routines (numpy's stable sort and linear quantile, bincount)
and to closed forms of the two update rules; planted mistakes must fail.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_balance.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv, src = line.split(";", 1)
        key, val = (s.strip() for s in kv.split("="))
        assert src.strip(), key
        vals[key] = float(val)
    return vals


def _logits(rng, T, E, ties=False):
    x = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        x = np.round(x * 2) / 2          # few distinct values: many equal scores
    return torch.from_numpy(x).to(torch.bfloat16)


def _ref_topk(logits, bias, k):
    x = logits.float().numpy()
    s = x + bias[None, :].astype(np.float32)          # binary32 add
    E = x.shape[1]
    out = np.empty((x.shape[0], k), dtype=np.int32)
    for t in range(x.shape[0]):
        order = np.lexsort((np.arange(E), -s[t]))      # score desc, then index asc
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("T,E,k,ties", [(50, 896, 8, False), (40, 64, 6, True), (7, 5, 5, True)])
def test_topk_matches_stable_sort(T, E, k, ties):
    rng = np.random.default_rng(T + E)
    x = _logits(rng, T, E, ties)
    bias = (0.1 * rng.standard_normal(E)).astype(np.float32)
    if ties:
        bias[:] = 0.0
    idx, sel, load = oracle.router_topk(x, bias, k)
    np.testing.assert_array_equal(idx, _ref_topk(x, bias, k))
    np.testing.assert_array_equal(load, np.bincount(idx.ravel(), minlength=E))
    np.testing.assert_array_equal(sel, np.take_along_axis(x.float().numpy(), idx, axis=1))


def test_load_accumulates_over_calls():
    rng = np.random.default_rng(1)
    x1, x2 = _logits(rng, 30, 40), _logits(rng, 20, 40)
    bias = np.zeros(40, np.float32)
    _, _, l1 = oracle.router_topk(x1, bias, 4)
    _, _, l12 = oracle.router_topk(x2, bias, 4, load=l1)
    _, _, both = oracle.router_topk(torch.cat([x1, x2]), bias, 4)
    np.testing.assert_array_equal(l12, both)
    assert l12.sum() == 50 * 4


@pytest.mark.parametrize("q", [0.0, 0.1, 0.25, 0.5, 0.75, 0.9, 1.0, 0.37])
def test_quantile_matches_numpy_linear(q):
    rng = np.random.default_rng(2)
    load = rng.integers(0, 5000, 896)
    _, (Qlo, Qhi) = oracle.router_update(load, np.zeros(896, np.float32), q_lo=q, q_hi=q)
    ref = float(np.quantile(load.astype(np.float64), q, method="linear"))
    assert Qlo == Qhi
    assert abs(Qhi - ref) <= 1e-12 * max(1.0, abs(ref))


def test_sign_update_closed_form_at_the_pages_quantiles():
    g = golden()
    E = int(g["experts"])
    rng = np.random.default_rng(3)
    load = rng.permutation(E).astype(np.int64) * 3 + 100        # distinct loads
    bias = (0.01 * rng.standard_normal(E)).astype(np.float32)
    eta = np.float32(1e-3)
    new, (Qlo, Qhi) = oracle.router_update(load, bias, "sign", g["q_lo_two_sided"],
                                           g["q_hi_two_sided"], eta)
    srt = np.sort(load)
    assert Qhi == float(np.quantile(srt, g["q_hi_two_sided"]))
    up, down = load < Qlo, load > Qhi
    # with distinct loads, the fraction above Q(0.9) is about 10 %
    assert abs(down.sum() - 0.1 * E) <= 1 and abs(up.sum() - 0.1 * E) <= 1
    ref = bias.copy()
    ref[down] = ref[down] - eta
    ref[up] = ref[up] + eta
    np.testing.assert_array_equal(new, ref)
    # the single-threshold median form moves every expert but the middle ones
    new, (m1, m2) = oracle.router_update(load, bias, "sign", g["q_single"], g["q_single"], eta)
    assert m1 == m2 == float(np.median(load))
    assert int((new != bias).sum()) == E - int((load == m1).sum())


def test_proportional_update_closed_form():
    g = golden()
    rng = np.random.default_rng(4)
    load = rng.integers(10, 1000, 896)
    bias = np.zeros(896, np.float32)
    new, (_, Q) = oracle.router_update(load, bias, "proportional", q_hi=g["q_proportional"],
                                       eta=0.01)
    np.testing.assert_allclose(new, 0.01 * (Q - load) / Q, rtol=1e-6, atol=1e-9)
    assert np.all((new < 0) == (load > Q)) and np.all((new > 0) == (load < Q))


def test_balanced_load_leaves_bias_unchanged():
    bias = np.linspace(-1, 1, 64).astype(np.float32)
    load = np.full(64, 123)
    for mode in ("sign", "proportional"):
        new, (a, b) = oracle.router_update(load, bias, mode, 0.1, 0.9, 0.5)
        assert a == b == 123.0
        np.testing.assert_array_equal(new, bias)


ROUTER_MUTANTS = {
    "ties_to_higher_index": ("if (best < 0 || s[e] > s[best]) best = e;",
                             "if (best < 0 || s[e] >= s[best]) best = e;"),
    "quantile_no_interpolation": ("return (double)xs[i] + (p - (double)i) * ((double)xs[j] - (double)xs[i]);",
                                  "return (double)xs[i];"),
    "sign_update_flipped": ("if (l > Qhi) bias[e] = bias[e] - eta;", "if (l > Qhi) bias[e] = bias[e] + eta;"),
    "proportional_over_load": ("(Qhi - l) / Qhi", "(Qhi - l) / l"),
    "bias_not_in_score": ("logit_at(logits, dtype, t * E + e) + bias[e];", "logit_at(logits, dtype, t * E + e);"),
}


@pytest.mark.parametrize("name", list(ROUTER_MUTANTS))
def test_router_mutant_is_rejected(tmp_path, name):
    old, new = ROUTER_MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "router_oracle.c")).read()
    assert src.count(old) == 1, name
    c, so = tmp_path / f"{name}.c", tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(c), "-lm"],
                   check=True)
    caught = False
    rng = np.random.default_rng(9)
    x = _logits(rng, 40, 64, ties=True)
    bias = (0.25 * rng.integers(-2, 3, 64)).astype(np.float32)
    idx, _, _ = oracle.router_topk(x, bias, 6, _lib_path=str(so))
    caught |= not np.array_equal(idx, _ref_topk(x, bias, 6))
    load = rng.integers(0, 500, 100)
    for mode in ("sign", "proportional"):
        new, (_, Q) = oracle.router_update(load, np.zeros(100, np.float32), mode, 0.37, 0.37, 0.01,
                                           _lib_path=str(so))
        ref_q = float(np.quantile(load.astype(np.float64), 0.37))
        caught |= abs(Q - ref_q) > 1e-9
        if mode == "sign":
            ref = np.where(load > ref_q, -0.01, np.where(load < ref_q, 0.01, 0.0)).astype(np.float32)
            caught |= not np.allclose(new, ref, atol=1e-7)
        else:
            caught |= not np.allclose(new, 0.01 * (ref_q - load) / ref_q, rtol=1e-6, atol=1e-9)
    assert caught
