"""Planted mistakes in copies of the oracle's C source must fail the pins.

Each mutant is a one-token edit of gdr_oracle.c (compiled into a temporary
directory, never into the package).  A pin battery -- the brute-force dense
product expansion and the beta = 0 closed form -- must reject every mutant,
which shows the pins can see a dropped term, a flipped sign, a swapped
operand, a transposed index or a wrong gate.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import chunk_ref
from test_oracle_pins import _brute_force, _case

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")

MUTANTS = {
    "drop_decay_in_prediction": ("p *= alpha;", ""),
    "flip_delta_sign": ("bt * (vj - p)", "bt * (vj + p)"),
    "output_reads_k": ("o += hij * qt[i];", "o += hij * kt[i];"),
    "drop_state_decay": ("const double hij = alpha * Hs[i * CB + c]", "const double hij = Hs[i * CB + c]"),
    "gate_argument": ("return -b * sigmoid(a);", "return -b * sigmoid(-a);"),
    "h0_transposed": ("h0[(((int64_t)n * H + h) * dk + i) * dv + j0 + c]",
                      "h0[(((int64_t)n * H + h) * dv + j0 + c) * dk + i]"),
    "erase_uses_q": ("p += Hs[i * CB + c] * kt[i];", "p += Hs[i * CB + c] * qt[i];"),
}


def _battery(path):
    """True if every pin passes for the build at ``path``."""
    rng = np.random.default_rng(123)
    q, k, v, a, beta, h0 = _case(rng, 9, dk=6, dv=6)
    out, hT = oracle.oracle_fwd(q, k, v, a, beta, h0=h0, b=2.0, _lib_path=path)
    g = chunk_ref.gate(a[0, :, 0], 2.0)
    ro, rh = _brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g, beta[0, :, 0], h0[0, 0])
    ok = np.allclose(out[0, :, 0], ro, rtol=1e-10, atol=1e-12) and \
        np.allclose(hT[0, 0], rh, rtol=1e-10, atol=1e-12)
    beta0 = np.zeros_like(beta)
    o0, _ = oracle.oracle_fwd(q, k, v, a, beta0, h0=h0, b=2.0, _lib_path=path)
    cg = np.cumsum(g)
    ok = ok and np.allclose(o0[0, :, 0], np.exp(cg)[:, None] * (q[0, :, 0] @ h0[0, 0]),
                            rtol=1e-11, atol=1e-13)
    return bool(ok)


def _compile(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(lib),
                    str(src), "-lm"], check=True)
    return str(lib)


def test_unmodified_source_passes(tmp_path):
    with open(SRC) as f:
        assert _battery(_compile(tmp_path, "orig", f.read()))


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_rejected(tmp_path, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    assert not _battery(_compile(tmp_path, name, text.replace(old, new)))
