"""GPU parity of the backward pass gdr_chunk_bwd against the fp64 oracle backward.

The gradients are those of L = <dout, out> + <dhT, hT> for the recurrence of
"Evaluating Next-Gen Sparse MoE and Long-Context LLMs" §2.2 (the oracle's
adjoint recurrence is pinned by finite differences of the forward oracle).
Tolerances, per gradient tensor: fp32 rel-L2 <= 1e-4; bf16 rel-L2 <= 1e-2 and
max-abs <= 5e-2 * max(1, max |ref|) (the outputs are rounded to bf16, 2^-9
relative, and each sum runs over up to 128 x 128 fp32 products).
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import rel_l2, to64

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "da", "dbeta", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _inputs(dtype, d, T, gate, seed, N=2, H=3, varlen=False, h0=True, a_mean=0.0):
    w = WORKLOADS["b2_t4k"].with_(B=N, H=H, dk=d, dv=d, dtype=dtype, h0_std=0.05 if h0 else 0.0,
                                  gate=gate, a_std=3.0 if gate == "softplus" else 1.0, seed=seed,
                                  varlen=varlen, a_mean=a_mean)
    x = make_inputs(w, device="cuda", T=T)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    B, Tn = x["q"].shape[:2]
    Ns = B if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1
    x["dout"] = torch.randn((B, Tn, H, d), generator=g).to(x["q"].dtype).cuda()
    x["dhT"] = (0.1 * torch.randn((Ns, H, d, d), generator=g)).cuda()
    return x


def _check(got, ref, dtype):
    for name in NAMES:
        if got[name] is None:
            continue
        x, r = to64(got[name]), ref[name]
        rl = rel_l2(x, r)
        if dtype == "f32":
            assert rl <= 1e-4, f"{name}: rel-L2 {rl:.3e}"
        else:
            assert rl <= 1e-2, f"{name}: rel-L2 {rl:.3e}"
            m = float(np.abs(x - r).max()) if r.size else 0.0
            lim = 5e-2 * max(1.0, float(np.abs(r).max()) if r.size else 0.0)
            assert m <= lim, f"{name}: max-abs {m:.3e} > {lim:.3e}"


def _run(x, gate, dout=True, dhT=True, h0=True, want_dh0=True):
    res = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"],
                        dout=x["dout"] if dout else None, dhT=x["dhT"] if dhT else None,
                        h0=x["h0"] if h0 else None, cu_seqlens=x["cu_seqlens"], b=x["b"],
                        gate=gate, want_dh0=want_dh0)
    torch.cuda.synchronize()
    st = gdr.gdr_get_status()
    assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
    ref = oracle.oracle_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"],
                            dout=x["dout"] if dout else None, dhT=x["dhT"] if dhT else None,
                            h0=x["h0"] if h0 else None, cu_seqlens=cu, b=x["b"], gate=gate)
    return dict(zip(NAMES, res)), ref


@pytest.mark.parametrize("dtype,d,gate", [("bf16", 128, "bounded"), ("f32", 64, "softplus"),
                                          ("f32", 128, "bounded"), ("bf16", 64, "softplus")])
def test_backward_matches_oracle(dtype, d, gate):
    # 77 tokens: four full 16-token checkpoint intervals and a ragged tail of 13
    x = _inputs(dtype, d, 77, gate, seed=4000 + d)
    got, ref = _run(x, gate)
    _check(got, ref, dtype)


def test_backward_packed_sequences():
    """Packed sequences of ragged lengths, one empty: dh0 of the empty one is its dhT."""
    x = _inputs("bf16", 128, 211, "bounded", seed=4100, N=1, H=2)
    x["cu_seqlens"] = torch.tensor([0, 5, 5, 40, 123, 211], dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(4101)
    x["h0"] = (0.05 * torch.randn((5, 2, 128, 128), generator=g)).cuda()
    x["dhT"] = (0.1 * torch.randn((5, 2, 128, 128), generator=g)).cuda()
    got, ref = _run(x, "bounded")
    _check(got, ref, "bf16")
    assert torch.equal(got["dh0"][1], x["dhT"][1])


@pytest.mark.parametrize("dout,dhT,h0", [(True, False, False), (False, True, True),
                                         (True, True, False)])
def test_backward_optional_arguments(dout, dhT, h0):
    x = _inputs("f32", 64, 40, "bounded", seed=4200)
    got, ref = _run(x, "bounded", dout=dout, dhT=dhT, h0=h0)
    _check(got, ref, "f32")


def test_backward_without_dh0_and_determinism():
    x = _inputs("bf16", 128, 50, "bounded", seed=4300)
    a, _ = _run(x, "bounded", want_dh0=False)
    b, _ = _run(x, "bounded", want_dh0=False)
    assert a["dh0"] is None
    for name in NAMES[:-1]:
        assert torch.equal(a[name], b[name]), name


def test_backward_zero_tokens_and_bad_args():
    x = _inputs("bf16", 128, 1, "bounded", seed=4400)
    empty = {n: x[n][:, :0] for n in ("q", "k", "v", "a", "beta", "dout")}
    dh0 = torch.full_like(x["dhT"], 7.0)
    outs = [torch.empty_like(empty[n]) for n in ("q", "k", "v", "a", "beta")]
    rc = gdr.gdr_chunk_bwd(empty["q"], empty["k"], empty["v"], empty["a"], empty["beta"], x["h0"],
                           empty["dout"], x["dhT"], *outs, dh0, None, 2, 0, 3, 128, 128, 16, 2.0,
                           gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED)
    assert rc == gdr.GDR_OK
    torch.cuda.synchronize()
    assert torch.equal(dh0, x["dhT"])
    outs = [torch.empty_like(x[n]) for n in ("q", "k", "v", "a", "beta")]
    base = [x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], x["dout"], x["dhT"]]
    assert gdr.gdr_chunk_bwd(*base, *outs, None, None, 2, 1, 3, 96, 128, 16, 2.0, gdr.GDR_BF16,
                             gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_bwd(*base, *outs, None, None, 2, 1, 3, 128, 128, 16, -1.0, gdr.GDR_BF16,
                             gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_INVALID_ARG
    aliased = [x["q"]] + outs[1:]   # dq on top of q
    assert gdr.gdr_chunk_bwd(*base, *aliased, None, None, 2, 1, 3, 128, 128, 16, 2.0,
                             gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED) == gdr.GDR_ERR_INVALID_ARG


@pytest.mark.parametrize("T,N,H,h0", [(300, 2, 2, True), (1000, 1, 2, False), (17, 3, 4, True)])
def test_chunked_backward_matches_oracle(T, N, H, h0):
    """bf16, d = 128, bounded gate: the chunked tensor-core form (forward state chain,
    adjoint chain, per-tile gradients), over many tiles and a ragged tail."""
    x = _inputs("bf16", 128, T, "bounded", seed=4600 + T, N=N, H=H, h0=h0)
    got, ref = _run(x, "bounded", h0=h0)
    _check(got, ref, "bf16")


def test_chunked_and_token_forms_agree(monkeypatch):
    """The same bf16 call through the chunked form and the token-by-token form."""
    x = _inputs("bf16", 128, 200, "bounded", seed=4700)
    chunked, ref = _run(x, "bounded")
    monkeypatch.setenv("GDR_BWD_TOKEN", "1")
    token, _ = _run(x, "bounded")
    for name in NAMES:
        r = rel_l2(to64(chunked[name]), to64(token[name]))
        assert r <= 1e-2, f"{name}: chunked vs token rel-L2 {r:.3e}"
    _check(chunked, ref, "bf16")
    _check(token, ref, "bf16")


@pytest.mark.parametrize("T,a_mean", [(2500, 0.0), (1500, -6.0), (5500, -6.0)])
def test_chunked_backward_segments(T, a_mean):
    """Long sequences: 64-tile segments of both state chains started at warm-up tiles
    (2500 tokens); a weak decay whose warm-ups run to the sequence ends (1500
    tokens); a weak decay with no warm-up within 256 tiles, run unsegmented (5500)."""
    x = _inputs("bf16", 128, T, "bounded", seed=4800 + T, N=1, H=2, a_mean=a_mean)
    got, ref = _run(x, "bounded")
    _check(got, ref, "bf16")


@pytest.mark.parametrize("T,a_mean,h0", [(2500, 0.0, True), (1500, -6.0, False), (77, 0.0, True)])
@pytest.mark.parametrize("chains", [("GDR_BWD_ADJ_MMA", "GDR_BWD_FWD_MMA"), ("GDR_BWD_ADJ_MMA",),
                                    ("GDR_BWD_FWD_MMA",)])
def test_chain_kernels_agree(monkeypatch, T, a_mean, h0, chains):
    """The state chains on tcgen05 (the default) and on mma.sync (GDR_BWD_ADJ_MMA=1 for
    the adjoint chain, GDR_BWD_FWD_MMA=1 for the forward chain): both match the oracle,
    and they agree with each other within the bf16 tolerance."""
    x = _inputs("bf16", 128, T, "bounded", seed=4900 + T, N=2, H=2, a_mean=a_mean, h0=h0)
    tc, ref = _run(x, "bounded", h0=h0)
    for name in chains:
        monkeypatch.setenv(name, "1")
    mma, _ = _run(x, "bounded", h0=h0)
    _check(tc, ref, "bf16")
    _check(mma, ref, "bf16")
    for name in NAMES:
        r = rel_l2(to64(tc[name]), to64(mma[name]))
        assert r <= 1e-2, f"{name}: tcgen05 vs mma.sync chains rel-L2 {r:.3e}"


@pytest.mark.parametrize("dout,dhT", [(False, True), (True, False)])
def test_chunked_backward_optional_arguments(dout, dhT):
    """bf16, d = 128 (the chunked form): dout = NULL (zero) and dhT = NULL (zero)."""
    x = _inputs("bf16", 128, 700, "bounded", seed=4950, N=2, H=2)
    got, ref = _run(x, "bounded", dout=dout, dhT=dhT)
    _check(got, ref, "bf16")


def test_chunked_backward_unaligned_inputs_take_the_token_form():
    """q one element off a 16-byte boundary: the call runs token by token (its tile
    kernel moves whole 16-byte pieces) and still matches the oracle."""
    x = _inputs("bf16", 128, 200, "bounded", seed=4960, N=1, H=2)
    big = torch.empty(x["q"].numel() + 1, dtype=x["q"].dtype, device="cuda")
    big[1:].copy_(x["q"].reshape(-1))
    x["q"] = big[1:].view(x["q"].shape)
    assert x["q"].data_ptr() % 16 != 0
    got, ref = _run(x, "bounded")
    _check(got, ref, "bf16")
