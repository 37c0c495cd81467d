"""GPU parity of the per-channel decay backward gdr_chunk_bwd_vec against the fp64
oracle ``oracle_bwd_vec`` (pinned by finite differences of the per-channel forward).

Each key channel of the state decays by its own factor exp(-b sigmoid(a_{t,i}))
("Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs", §2.1-2.2);
the gradients are those of <dout, out> + <dhT, hT>, with da one value per channel.
Tolerances as for the scalar backward: rel-L2 <= 1e-2 and max-abs <= 5e-2 max(1, |ref|).
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_channel_gate, make_inputs
from gpu_helpers import rel_l2, to64

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "da", "dbeta", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _inputs(T, seed, N=2, H=3, a_mean=0.0, h0=True):
    w = WORKLOADS["b2_t4k"].with_(B=N, H=H, h0_std=0.05 if h0 else 0.0, seed=seed)
    x = make_inputs(w, device="cuda", T=T)
    x["av"] = make_channel_gate(x, seed + 7, a_mean=a_mean)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    Ns = N if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1
    x["dout"] = torch.randn(x["v"].shape, generator=g).to(torch.bfloat16).cuda()
    x["dhT"] = (0.1 * torch.randn((Ns, H, 128, 128), generator=g)).cuda()
    return x


def _check(got, ref):
    for name in NAMES:
        x, r = to64(got[name]), ref[name]
        rl = rel_l2(x, r)
        assert rl <= 1e-2, f"{name}: rel-L2 {rl:.3e}"
        lim = 5e-2 * max(1.0, float(np.abs(r).max()) if r.size else 0.0)
        assert float(np.abs(x - r).max()) <= lim, f"{name}: max-abs"


def _run(x):
    got = gdr.chunk_bwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], dout=x["dout"],
                            dhT=x["dhT"], h0=x["h0"], cu_seqlens=x["cu_seqlens"], b=2.0)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
    ref = oracle.oracle_bwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], dout=x["dout"],
                                dhT=x["dhT"], h0=x["h0"], cu_seqlens=cu, b=2.0)
    return dict(zip(NAMES, got)), ref


@pytest.mark.parametrize("T,N,H", [(77, 2, 3), (300, 1, 2), (16, 3, 2)])
def test_vec_backward_matches_oracle(T, N, H):
    x = _inputs(T, seed=7000 + T, N=N, H=H)
    got, ref = _run(x)
    _check(got, ref)


def test_vec_backward_packed_and_segmented():
    """Packed sequences with one empty, and a 2500-token sequence run in segments."""
    x = _inputs(2600, seed=7100, N=1, H=2)
    x["cu_seqlens"] = torch.tensor([0, 9, 9, 100, 2600], dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(7101)
    x["h0"] = (0.05 * torch.randn((4, 2, 128, 128), generator=g)).cuda()
    x["dhT"] = (0.1 * torch.randn((4, 2, 128, 128), generator=g)).cuda()
    got, ref = _run(x)
    _check(got, ref)
    assert torch.equal(got["dh0"][1], x["dhT"][1])


def test_vec_backward_equal_channels_match_scalar_backward():
    x = _inputs(200, seed=7200)
    x["av"] = x["a"][..., None].expand(*x["a"].shape, 128).contiguous()
    v = gdr.chunk_bwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], dout=x["dout"], dhT=x["dhT"],
                          h0=x["h0"], b=2.0)
    s = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], dout=x["dout"], dhT=x["dhT"],
                      h0=x["h0"], b=2.0)
    torch.cuda.synchronize()
    for name, gv, gs in zip(NAMES, v, s):
        if name == "da":
            gv = gv.float().sum(dim=-1)
        assert rel_l2(to64(gv), to64(gs)) <= 1e-2, name


def test_vec_backward_rejects_what_it_does_not_cover():
    x = _inputs(16, seed=7300)
    outs = [torch.empty_like(x[n]) for n in ("q", "k", "v", "av", "beta")]
    base = [x["q"], x["k"], x["v"], x["av"], x["beta"], x["h0"], x["dout"], x["dhT"], *outs, None,
            None, 2, 16, 3, 128, 128]
    assert gdr.gdr_chunk_bwd_vec(*base, 32, 2.0, gdr.GDR_BF16) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_bwd_vec(*base, 16, 6.0, gdr.GDR_BF16) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_bwd_vec(*base, 16, 2.0, gdr.GDR_F32) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_bwd_vec(*base, 16, -1.0, gdr.GDR_BF16) == gdr.GDR_ERR_INVALID_ARG


@pytest.mark.parametrize("T,a_mean", [(2500, 0.0), (600, -6.0)])
def test_vec_chain_kernels_agree(monkeypatch, T, a_mean):
    """Per-channel decay: the state chains on tcgen05 (the default) and on mma.sync
    (GDR_BWD_ADJ_MMA=1, GDR_BWD_FWD_MMA=1) both match the oracle and agree."""
    x = _inputs(T, seed=7400 + T, N=2, H=2, a_mean=a_mean)
    tc, ref = _run(x)
    monkeypatch.setenv("GDR_BWD_ADJ_MMA", "1")
    monkeypatch.setenv("GDR_BWD_FWD_MMA", "1")
    mma, _ = _run(x)
    _check(tc, ref)
    _check(mma, ref)
    for name in NAMES:
        r = rel_l2(to64(tc[name]), to64(mma[name]))
        assert r <= 1e-2, f"{name}: tcgen05 vs mma.sync chains rel-L2 {r:.3e}"


def test_vec_backward_without_dout():
    """dout = NULL (zero) on the per-channel chunked form."""
    x = _inputs(500, seed=7500, N=1, H=2)
    got = gdr.chunk_bwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], dout=None, dhT=x["dhT"],
                            h0=x["h0"], b=2.0)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    ref = oracle.oracle_bwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], dout=None, dhT=x["dhT"],
                                h0=x["h0"], b=2.0)
    _check(dict(zip(NAMES, got)), ref)
