"""Full-size parity: the workloads at their stated sizes, in the launch
configuration the benchmark times (automatic path, tile 16 where given), checked
against the fp64 oracle on outputs it can compute in seconds.

* 1M-token single sequence: a seeded 8192-token slice of the outputs, the state
  entering that slice, and the final state, for a seeded sample of two heads.
  The oracle runs the slice from the GPU's entering state (a prefix call's hT);
  that entering state is compared separately with the oracle's own state at the
  slice start; the final state with the oracle's full-length run.
* packed varlen batch (1M tokens): every output and final state of two sampled
  heads, with the bounded gate and with the unbounded softplus gate; the
  relative L2 error of each is printed (the divergence report).
* 32-head, 64K-token sweep over tile {16, 32, 64} x bound {2, 8}: every output
  and final state of four sampled heads.

Tolerances as everywhere for bf16: rel-L2 <= 1e-2 and max-abs <= 5e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from gdr_inputs import WORKLOADS, h32_variant, make_inputs, softplus_variant
from gpu_helpers import assert_close, rel_l2, run_gpu, to64

pytestmark = pytest.mark.gpu

SLICE = 8192
ORACLE_BLOCK = 1 << 17      # oracle tokens per call (bounds its fp64 output buffer)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _heads_cpu(x, heads, t0, t1):
    """q, k, v, a, beta of tokens [t0, t1) and the given heads, on the host."""
    idx = torch.tensor(heads, device=x["q"].device)
    return [x[n][:, t0:t1].index_select(2, idx).contiguous().cpu()
            for n in ("q", "k", "v", "a", "beta")]


def _oracle_run(x, heads, t0, t1, h0, b, gate, keep_out=True):
    """The oracle over tokens [t0, t1) of one sequence for the given heads,
    in blocks chained through the state; returns (out or None, state)."""
    outs = []
    h = h0
    for s in range(t0, t1, ORACLE_BLOCK):
        e = min(t1, s + ORACLE_BLOCK)
        q, k, v, a, beta = _heads_cpu(x, heads, s, e)
        o, h = oracle.oracle_fwd(q, k, v, a, beta, h0=h, b=b, gate=gate)
        if keep_out:
            outs.append(o)
    return (np.concatenate(outs, axis=1) if keep_out else None), h


def test_t1m_slice_entering_and_final_state():
    w = WORKLOADS["t1m"]
    x = make_inputs(w, device="cuda")
    T, H = x["T"], x["H"]
    out, hT = run_gpu(x)
    rng = np.random.default_rng(w.seed)
    s0 = 16 * int(rng.integers(1, (T - SLICE) // 16))
    heads = sorted(int(h) for h in rng.choice(H, size=2, replace=False))
    # the GPU state entering the slice: a prefix call (the h0 -> hT carry)
    xp = dict(x, q=x["q"][:, :s0], k=x["k"][:, :s0], v=x["v"][:, :s0], a=x["a"][:, :s0],
              beta=x["beta"][:, :s0], T=s0)
    _, h_enter = run_gpu(xp)
    h_enter_heads = to64(h_enter[:, heads])
    # oracle: its own state at s0, the slice from the GPU's state, and the end
    _, h_ref_s0 = _oracle_run(x, heads, 0, s0, None, w.b, w.gate, keep_out=False)
    assert_close(h_enter_heads, h_ref_s0, "bf16", f"state entering token {s0}")
    o_slice, _ = _oracle_run(x, heads, s0, s0 + SLICE, h_enter_heads, w.b, w.gate)
    got = to64(out[:, s0:s0 + SLICE][:, :, heads])
    assert_close(got, o_slice, "bf16", f"out[{s0}:{s0 + SLICE}] heads {heads}")
    _, h_ref_T = _oracle_run(x, heads, s0, T, h_ref_s0, w.b, w.gate, keep_out=False)
    assert_close(to64(hT[:, heads]), h_ref_T, "bf16", "final state")


@pytest.mark.parametrize("softplus", [False, True])
def test_varlen_1m_sampled_heads(softplus):
    w = WORKLOADS["varlen_1m"]
    if softplus:
        w = softplus_variant(w)
    x = make_inputs(w, device="cuda")
    out, hT = run_gpu(x)
    rng = np.random.default_rng(w.seed)
    heads = sorted(int(h) for h in rng.choice(x["H"], size=2, replace=False))
    cu = x["cu_seqlens"].cpu().tolist()
    h0 = x["h0"][:, heads].contiguous().cpu()
    num2 = den2 = 0.0
    mabs = 0.0
    h_ref = np.zeros((len(cu) - 1, len(heads), x["dk"], x["dv"]))
    for n in range(len(cu) - 1):
        o_ref, h_n = _oracle_run(x, heads, cu[n], cu[n + 1], h0[n:n + 1], w.b, w.gate)
        got = to64(out[:, cu[n]:cu[n + 1]][:, :, heads])
        num2 += float(((got - o_ref) ** 2).sum())
        den2 += float((o_ref ** 2).sum())
        mabs = max(mabs, float(np.abs(got - o_ref).max()))
        h_ref[n] = h_n[0]
    r_out = (num2 / den2) ** 0.5
    r_hT = rel_l2(to64(hT[:, heads]), h_ref)
    print(f"\n[divergence] varlen_1m gate={w.gate}: out rel-L2 {r_out:.3e} max-abs {mabs:.3e}; "
          f"hT rel-L2 {r_hT:.3e} ({len(cu) - 1} sequences, heads {heads})")
    assert r_out <= 1e-2 and mabs <= 5e-2
    assert_close(to64(hT[:, heads]), h_ref, "bf16", "final states")


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("b", [2, 8])
def test_h32_t64k_sampled_heads(chunk, b):
    w = h32_variant(chunk, b)
    x = make_inputs(w, device="cuda")
    out, hT = run_gpu(x)
    rng = np.random.default_rng(w.seed)
    heads = sorted(int(h) for h in rng.choice(x["H"], size=4, replace=False))
    o_ref, h_ref = _oracle_run(x, heads, 0, x["T"], None, w.b, w.gate)
    r = assert_close(to64(out[:, :, heads]), o_ref, "bf16", "out")
    rh = assert_close(to64(hT[:, heads]), h_ref, "bf16", "hT")
    print(f"\n[divergence] {w.name}: out rel-L2 {r:.3e}, hT rel-L2 {rh:.3e}, heads {heads}")
