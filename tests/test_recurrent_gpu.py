"""GPU parity of the recurrent (decoding) form gdr_recurrent_fwd against the fp64
oracle, and prefill with the chunked form followed by token-by-token decoding.

The recurrence is the one of every other entry point ("Evaluating Next-Gen
Sparse MoE and Long-Context LLMs", §2.2): per token H <- alpha H + beta k (v -
alpha H^T k)^T and o = H^T q, with the state carried in place between calls.
Tolerances as elsewhere: fp32 rel-L2 <= 1e-4; bf16 rel-L2 <= 1e-2, max-abs <= 5e-2.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, run_gpu, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _inputs(dtype, d, T, gate, seed, N=3, H=4):
    w = WORKLOADS["b2_t4k"].with_(B=N, H=H, dk=d, dv=d, dtype=dtype, h0_std=0.05, gate=gate,
                                  a_std=3.0 if gate == "softplus" else 1.0, seed=seed)
    return make_inputs(w, device="cuda", T=T)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 64), ("f32", 128)])
@pytest.mark.parametrize("T", [1, 7])
@pytest.mark.parametrize("gate", ["bounded", "softplus"])
def test_recurrent_matches_oracle(dtype, d, T, gate):
    x = _inputs(dtype, d, T, gate, seed=3000 + 10 * T + d)
    state = x["h0"].clone()
    out = gdr.recurrent_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], state, b=x["b"], gate=gate)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    ro, rh = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"], b=x["b"],
                               gate=gate)
    assert_close(to64(out), ro, dtype, "out")
    assert_close(to64(state), rh, dtype, "state")


def test_prefill_then_decode_token_by_token():
    """Prefill 250 tokens with the chunked form (its hT is the state), then decode
    50 tokens with one call per token; the outputs and the final state equal the
    oracle's over all 300 tokens."""
    T0, T1 = 250, 50
    x = _inputs("bf16", 128, T0 + T1, "bounded", seed=3100, N=2, H=4)
    pre = {n: x[n][:, :T0].contiguous() for n in ("q", "k", "v", "a", "beta")}
    xp = dict(x, **pre, T=T0)
    out0, state = run_gpu(xp)
    outs = [out0]
    for t in range(T0, T0 + T1):
        step = {n: x[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "a", "beta")}
        outs.append(gdr.recurrent_fwd(step["q"], step["k"], step["v"], step["a"], step["beta"],
                                      state, b=x["b"]))
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    out = torch.cat(outs, dim=1)
    ro, rh = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"], b=x["b"])
    assert_close(to64(out), ro, "bf16", "out")
    assert_close(to64(state), rh, "bf16", "state")
    # the decode steps alone, against the oracle's outputs for those tokens
    assert_close(to64(out[:, T0:]), ro[:, T0:], "bf16", "decoded tokens")


def test_zero_tokens_leave_state_untouched_and_bad_args_are_rejected():
    x = _inputs("bf16", 128, 1, "bounded", seed=3200)
    state = x["h0"].clone()
    empty = {n: x[n][:, :0] for n in ("q", "k", "v", "a", "beta")}
    out = torch.empty((3, 0, 4, 128), dtype=torch.bfloat16, device="cuda")
    rc = gdr.gdr_recurrent_fwd(empty["q"], empty["k"], empty["v"], empty["a"], empty["beta"],
                               state, out, 3, 0, 4, 128, 128, 2.0, gdr.GDR_BF16,
                               gdr.GDR_GATE_BOUNDED)
    assert rc == gdr.GDR_OK
    torch.cuda.synchronize()
    assert torch.equal(state, x["h0"])
    out1 = torch.empty((3, 1, 4, 128), dtype=torch.bfloat16, device="cuda")
    args = [x["q"], x["k"], x["v"], x["a"], x["beta"], state, out1]
    assert gdr.gdr_recurrent_fwd(*args, 3, 1, 4, 96, 128, 2.0, gdr.GDR_BF16,
                                 gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_recurrent_fwd(*args, 3, 1, 4, 128, 128, -1.0, gdr.GDR_BF16,
                                 gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_INVALID_ARG
    assert gdr.gdr_recurrent_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], state, x["v"], 3, 1,
                                 4, 128, 128, 2.0, gdr.GDR_BF16,
                                 gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_INVALID_ARG
