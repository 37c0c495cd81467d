"""Pins of the oracle's backward pass (``oracle_bwd``).

The backward is checked against central finite differences of the forward
oracle (``oracle_fwd``, itself pinned by brute-force products and closed forms):
for L = <dout, out> + <dhT, hT> and a random direction R of one input X,
    (L(X + eps R) - L(X - eps R)) / (2 eps)  ~=  <dL/dX, R>.
One directional derivative per input covers every entry of its gradient (a
wrong term anywhere shifts it), so each case checks q, k, v, a, beta and h0.
The cases cross the oracle's 64-token checkpoints and include packed sequences
(one of them empty) and both gate forms.  All in fp64 on the CPU.
"""
import numpy as np
import pytest

import oracle


def _case(rng, B, T, H, dk, dv, varlen=False):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk)) / np.sqrt(dk)
    v = rng.standard_normal((B, T, H, dv))
    a = rng.standard_normal((B, T, H))
    beta = rng.uniform(0.1, 0.9, (B, T, H))
    cu = None
    N = B
    if varlen:
        cu = np.array([0, 3, 3, T // 2, T], dtype=np.int64)
        N = len(cu) - 1
    h0 = 0.3 * rng.standard_normal((N, H, dk, dv))
    dout = rng.standard_normal((B, T, H, dv))
    dhT = rng.standard_normal((N, H, dk, dv))
    return dict(q=q, k=k, v=v, a=a, beta=beta, h0=h0), cu, dout, dhT


def _loss(x, cu, dout, dhT, b, gate):
    out, hT = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"],
                                cu_seqlens=cu, b=b, gate=gate)
    return float((out * dout).sum() + (hT * dhT).sum())


@pytest.mark.parametrize("B,T,H,dk,dv,varlen,gate,b", [
    (2, 7, 2, 3, 4, False, "bounded", 2.0),
    (1, 9, 1, 4, 3, False, "softplus", 2.0),
    (1, 150, 1, 3, 2, False, "bounded", 5.0),      # crosses two checkpoints
    (1, 40, 2, 3, 3, True, "bounded", 2.0),        # packed, with an empty sequence
    (1, 131, 1, 2, 3, True, "softplus", 2.0),
])
def test_backward_matches_finite_differences(B, T, H, dk, dv, varlen, gate, b):
    rng = np.random.default_rng(7 + T + dk)
    x, cu, dout, dhT = _case(rng, B, T, H, dk, dv, varlen)
    g = oracle.oracle_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], dout=dout, dhT=dhT,
                          h0=x["h0"], cu_seqlens=cu, b=b, gate=gate)
    grads = {"q": g["dq"], "k": g["dk"], "v": g["dv"], "a": g["da"], "beta": g["dbeta"],
             "h0": g["dh0"]}
    eps = 1e-5
    for name, grad in grads.items():
        R = rng.standard_normal(x[name].shape)
        xp = dict(x, **{name: x[name] + eps * R})
        xm = dict(x, **{name: x[name] - eps * R})
        fd = (_loss(xp, cu, dout, dhT, b, gate) - _loss(xm, cu, dout, dhT, b, gate)) / (2 * eps)
        an = float((grad * R).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_zero_upstream_gives_zero_gradients():
    rng = np.random.default_rng(3)
    x, cu, dout, dhT = _case(rng, 1, 20, 2, 3, 3)
    g = oracle.oracle_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"])
    for name, arr in g.items():
        assert not np.any(arr), name


def test_state_gradient_passes_through_pure_decay():
    """beta = 0 and dout = 0: hT = e^{sum g} h0, so dh0 = e^{sum g} dhT exactly and
    dq = dk = dv = 0."""
    rng = np.random.default_rng(4)
    x, cu, dout, dhT = _case(rng, 1, 30, 1, 3, 3)
    x["beta"] = np.zeros_like(x["beta"])
    g = oracle.oracle_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], dhT=dhT, h0=x["h0"])
    decay = np.exp(sum(oracle.gate(z, 2.0) for z in x["a"][0, :, 0]))
    np.testing.assert_allclose(g["dh0"], decay * dhT, rtol=1e-12, atol=0)
    for name in ("dq", "dk", "dv"):
        assert not np.any(g[name]), name


# One-token edits of the backward in gdr_oracle.c; the finite-difference pin
# must reject each (a dropped term, a wrong operand, a flipped sign).
BWD_MUTANTS = {
    "drop_k_through_prediction": ("g_k += alpha * Hp[i * dv + j] * dp[j];", ""),
    "decay_grad_reads_new_state": ("dalpha += Hp[i * dv + j] * dhb;", "dalpha += Ht[i * dv + j] * dhb;"),
    "beta_grad_sign": ("dbt += acc * (widen(v, in_dtype, row * dv + j) - p[j]);",
                       "dbt += acc * (widen(v, in_dtype, row * dv + j) + p[j]);"),
    "output_grad_uses_k": ("dH[i * dv + j] += qt[i] * g_o;", "dH[i * dv + j] += kt[i] * g_o;"),
    "state_grad_not_decayed": ("dH[i * dv + j] = alpha * dhb;", "dH[i * dv + j] = dhb;"),
}


@pytest.mark.parametrize("name", list(BWD_MUTANTS))
def test_backward_mutant_is_rejected(tmp_path, name):
    import os
    import subprocess
    old, new = BWD_MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")).read()
    assert src.count(old) == 1
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(c),
                    "-lm"], check=True)
    rng = np.random.default_rng(11)
    x, cu, dout, dhT = _case(rng, 2, 7, 2, 3, 4)
    g = oracle.oracle_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], dout=dout, dhT=dhT,
                          h0=x["h0"], _lib_path=str(so))
    grads = {"q": g["dq"], "k": g["dk"], "v": g["dv"], "a": g["da"], "beta": g["dbeta"],
             "h0": g["dh0"]}
    eps, caught = 1e-5, False
    for xname, grad in grads.items():
        R = rng.standard_normal(x[xname].shape)
        fd = (_loss(dict(x, **{xname: x[xname] + eps * R}), cu, dout, dhT, 2.0, "bounded")
              - _loss(dict(x, **{xname: x[xname] - eps * R}), cu, dout, dhT, 2.0, "bounded")) / (2 * eps)
        caught |= abs(fd - float((grad * R).sum())) > 1e-6 * max(1.0, abs(fd))
    assert caught
