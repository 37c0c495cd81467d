"""The Python binding checks the tensors of its tensor-level calls before the C call
(CPU only: no compute call runs here).

The C entry points take pointers and sizes, so they cannot see a tensor of the wrong
shape, dtype, device or layout.  The binding takes the sizes from q (or the router
logits) and refuses any other tensor that disagrees, and any tensor that is not on a
CUDA device, with ValueError, before calling into the library.  The layouts the
library's own tests and benchmark pass (every workload recipe, packed sequences,
per-channel gates, gradients, decode slices) must all be accepted.
"""
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
from gdr_inputs import WORKLOADS, make_channel_gate, make_inputs, make_router_logits


def _small(name, T=40, **kw):
    return make_inputs(WORKLOADS[name].with_(**kw), device="cpu", T=T)


def _args(x):
    return [x[n] for n in ("q", "k", "v", "a", "beta")]


# ---- accepted: the layouts the tests and the benchmark use -----------------------------
@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_every_workload_recipe_is_accepted(name):
    x = _small(name, H=2)
    B, T, H, dk, dv, N = gdr.check_sequence_inputs(*_args(x), h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    assert (B, T, H) == tuple(x["q"].shape[:3]) and dk == x["q"].shape[-1] and dv == x["v"].shape[-1]
    assert N == (B if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1)


def test_packed_sequences_with_states_and_gradients_are_accepted():
    x = _small("b2_t4k", T=211, B=1, H=2)
    cu = torch.tensor([0, 5, 5, 40, 123, 211], dtype=torch.int32)
    h0 = torch.zeros((5, 2, 128, 128))
    dhT = torch.zeros((5, 2, 128, 128))
    dout = torch.zeros_like(x["v"])
    assert gdr.check_sequence_inputs(*_args(x), h0=h0, cu_seqlens=cu, dout=dout, dhT=dhT)[-1] == 5


def test_per_channel_gate_and_decode_slices_are_accepted():
    x = _small("b2_t4k", T=60, B=2, H=2)
    av = make_channel_gate(x, 7)
    gdr.check_sequence_inputs(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"], per_channel=True)
    step = [t[:, 10:11].contiguous() for t in _args(x)]
    state = x["h0"].clone()
    gdr.check_sequence_inputs(*step, h0=state, out=torch.empty_like(step[2]))
    empty = [t[:, :0] for t in _args(x)]          # zero tokens
    gdr.check_sequence_inputs(*empty, h0=state)


def test_fp32_and_mixed_widths_are_accepted():
    x = _small("small_fp32")
    gdr.check_sequence_inputs(*_args(x))
    x = _small("b2_t4k", H=2, dk=64, dv=128)
    assert gdr.check_sequence_inputs(*_args(x))[3:5] == (64, 128)


# ---- refused -----------------------------------------------------------------------------
def _bad(**change):
    x = _small("b2_t4k", B=2, H=2)
    kw = dict(q=x["q"], k=x["k"], v=x["v"], a=x["a"], beta=x["beta"], h0=x["h0"], cu_seqlens=None)
    kw.update(change)
    return kw


@pytest.mark.parametrize("what,change", [
    ("k tokens", lambda x: dict(k=x["k"][:, :-1])),
    ("k width", lambda x: dict(k=x["k"][..., :64].contiguous())),
    ("v heads", lambda x: dict(v=torch.zeros((2, 40, 3, 128), dtype=torch.bfloat16))),
    ("a per channel given to the scalar call", lambda x: dict(a=torch.zeros((2, 40, 2, 128), dtype=torch.bfloat16))),
    ("beta dtype", lambda x: dict(beta=x["beta"].float())),
    ("q dtype", lambda x: dict(q=x["q"].half())),
    ("h0 sequences", lambda x: dict(h0=x["h0"][:1])),
    ("h0 dtype", lambda x: dict(h0=x["h0"].double())),
    ("k not contiguous", lambda x: dict(k=x["k"].transpose(0, 1).contiguous().transpose(0, 1))),
    ("v on another device", lambda x: dict(v=torch.empty(x["v"].shape, dtype=x["v"].dtype, device="meta"))),
    ("cu_seqlens with B = 2", lambda x: dict(cu_seqlens=torch.tensor([0, 10, 40], dtype=torch.int32))),
    ("missing beta", lambda x: dict(beta=None)),
])
def test_mismatched_tensors_are_refused(what, change):
    x = _small("b2_t4k", B=2, H=2)
    kw = _bad(**change(x))
    with pytest.raises(ValueError):
        gdr.check_sequence_inputs(**kw)


def test_packed_offsets_must_be_int32_and_match_the_states():
    x = _small("b2_t4k", T=100, B=1, H=2)
    with pytest.raises(ValueError):
        gdr.check_sequence_inputs(*_args(x), cu_seqlens=torch.tensor([0, 50, 100]))   # int64
    cu = torch.tensor([0, 50, 100], dtype=torch.int32)
    with pytest.raises(ValueError):
        gdr.check_sequence_inputs(*_args(x), cu_seqlens=cu, h0=torch.zeros((3, 2, 128, 128)))
    with pytest.raises(ValueError):
        gdr.check_sequence_inputs(*_args(x), cu_seqlens=cu, dhT=torch.zeros((1, 2, 128, 128)))


def test_per_channel_call_needs_a_channel_gate():
    x = _small("b2_t4k", B=1, H=2)
    with pytest.raises(ValueError):
        gdr.check_sequence_inputs(*_args(x), per_channel=True)     # a is [B, T, H]


# ---- CPU tensors never reach the library -------------------------------------------------
def test_tensor_calls_refuse_cpu_tensors():
    x = _small("b2_t4k", B=1, H=2)
    for call in (lambda: gdr.chunk_fwd(*_args(x)),
                 lambda: gdr.chunk_bwd(*_args(x)),
                 lambda: gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], make_channel_gate(x, 3), x["beta"]),
                 lambda: gdr.recurrent_fwd(*_args(x), torch.zeros((1, 2, 128, 128)))):
        with pytest.raises(ValueError, match="CUDA"):
            call()
    logits, bias = make_router_logits(64, 32, 5, "bf16", device="cpu")
    with pytest.raises(ValueError, match="CUDA"):
        gdr.router_topk(logits, bias, 4)
    with pytest.raises(ValueError, match="CUDA"):
        gdr.router_bias_update(torch.zeros(32, dtype=torch.int64), bias)


def test_router_tensors_are_checked():
    logits, bias = make_router_logits(64, 32, 5, "bf16", device="cpu")
    with pytest.raises(ValueError):
        gdr.router_topk(logits, bias[:16], 4)                                  # bias length
    with pytest.raises(ValueError):
        gdr.router_topk(logits, bias, 4, load=torch.zeros(32, dtype=torch.int32))   # load dtype
    with pytest.raises(ValueError):
        gdr.router_bias_update(torch.zeros(16, dtype=torch.int64), bias)         # load length
    with pytest.raises(ValueError):
        gdr.router_bias_update(torch.zeros(32, dtype=torch.int64), bias, mode="median")
    with pytest.raises(ValueError):
        gdr.recurrent_fwd(*_args(_small("b2_t4k", B=1, H=2)), None)             # no state
