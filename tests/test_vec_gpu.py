"""GPU parity of the per-channel decay forward gdr_chunk_fwd_vec against the fp64
oracle ``oracle_fwd_vec``.

Each key channel i of the state decays by exp(-b sigmoid(a_{t,i})) before the
delta-rule write ("Deep Dive: The Next Generation of Ultra-Long Context Sparse
MoE LLMs", §2.1-2.2).  Tolerances as for the scalar form: fp32 rel-L2 <= 1e-4;
bf16 rel-L2 <= 1e-2 and max-abs <= 5e-2, on out and hT.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_channel_gate, make_inputs
from gpu_helpers import assert_close, run_gpu, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _inputs(dtype, d, T, seed, N=2, H=3, h0=True, b=2.0, a_std=1.0, varlen=False, a_mean=0.0):
    w = WORKLOADS["b2_t4k"].with_(B=N, H=H, dk=d, dv=d, dtype=dtype, h0_std=0.05 if h0 else 0.0,
                                  seed=seed, b=b, varlen=varlen, len_min=1, len_max=max(1, T // 3))
    x = make_inputs(w, device="cuda", T=T)
    x["av"] = make_channel_gate(x, seed + 7, a_std=a_std, a_mean=a_mean)
    return x


def _check(x, dtype, b=2.0):
    out, hT = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"],
                                cu_seqlens=x["cu_seqlens"], b=b)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
    ro, rh = oracle.oracle_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"],
                                   cu_seqlens=cu, b=b)
    assert_close(to64(out), ro, dtype, "out")
    assert_close(to64(hT), rh, dtype, "hT")
    return out, hT


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("f32", 128), ("bf16", 64)])
@pytest.mark.parametrize("T", [16, 100])
def test_vec_matches_oracle(dtype, d, T):
    _check(_inputs(dtype, d, T, seed=5000 + T + d), dtype)


def test_vec_packed_sequences_and_no_h0():
    x = _inputs("bf16", 128, 1000, seed=5100, N=1, H=4, h0=False, varlen=True)
    assert x["cu_seqlens"].numel() > 3
    _check(x, "bf16")


@pytest.mark.parametrize("b,a_std", [(5.0, 3.0), (0.5, 1.0)])
def test_vec_gate_bound_extremes(b, a_std):
    """b = 5 (the largest bound taken: exp(-G) up to exp(80) inside a tile) and a
    weak decay; fp32 keeps rel-L2 <= 1e-4 at both ends."""
    _check(_inputs("f32", 128, 160, seed=5200, b=b, a_std=a_std), "f32", b=b)


def test_vec_equal_channels_match_scalar_path():
    """All channels sharing a: the per-channel path and the scalar chunked path
    compute the same recurrence (both checked against the scalar oracle)."""
    x = _inputs("f32", 128, 200, seed=5300)
    x["av"] = x["a"][..., None].expand(*x["a"].shape, 128).contiguous()
    out_v, hT_v = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"], b=2.0)
    out_s, hT_s = run_gpu(x)
    ro, rh = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"], b=2.0)
    assert_close(to64(out_v), ro, "f32", "vec out")
    assert_close(to64(hT_v), rh, "f32", "vec hT")
    assert_close(to64(out_v), to64(out_s), "f32", "vec vs scalar out")


def test_vec_zero_tokens_and_bad_args():
    x = _inputs("bf16", 128, 16, seed=5400)
    hT = torch.full_like(x["h0"], 3.0)
    e = {n: x[n][:, :0] for n in ("q", "k", "v", "av", "beta")}
    out0 = torch.empty_like(e["v"])
    assert gdr.gdr_chunk_fwd_vec(e["q"], e["k"], e["v"], e["av"], e["beta"], x["h0"], out0, hT,
                                 None, 2, 0, 3, 128, 128, 16, 2.0, gdr.GDR_BF16) == gdr.GDR_OK
    torch.cuda.synchronize()
    assert torch.equal(hT, x["h0"])
    out = torch.empty_like(x["v"])
    args = [x["q"], x["k"], x["v"], x["av"], x["beta"], x["h0"], out, hT, None, 2, 16, 3, 128, 128]
    assert gdr.gdr_chunk_fwd_vec(*args, 32, 2.0, gdr.GDR_BF16) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_fwd_vec(*args, 16, 6.0, gdr.GDR_BF16) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_chunk_fwd_vec(*args, 16, -1.0, gdr.GDR_BF16) == gdr.GDR_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = x["av"]   # out on top of a
    assert gdr.gdr_chunk_fwd_vec(*bad, 16, 2.0, gdr.GDR_BF16) == gdr.GDR_ERR_INVALID_ARG


def test_vec_long_sequences_run_in_segments():
    """3000 tokens = 188 tiles: three 64-tile segments, the later two started from
    a zero state at a warm-up tile where the decay bound is below 2^-64."""
    _check(_inputs("bf16", 128, 3000, seed=5500, N=1, H=2), "bf16")


def test_vec_weak_decay_runs_unsegmented():
    """a ~ N(-6, 1) per channel: the weakest channel decays by about 1 - 0.005 per
    token, so no warm-up within 256 tiles reaches 2^-64 and the pair runs as one
    block from h0 (5000 tokens = 313 tiles)."""
    _check(_inputs("bf16", 128, 5000, seed=5600, N=1, H=2, a_mean=-6.0), "bf16")


def test_vec_one_failed_warm_up_runs_the_pair_unsegmented():
    """6000 tokens = 375 tiles in 64-tile segments.  Head 0 has a weak decay on tokens
    1024-5119 (tiles 64-319), so the walk back from the segment start at tile 320 finds
    no warm-up within 256 tiles: head 0 runs as one block.  Its other segment starts
    (tiles 64-256) could reach the sequence start, and head 1 decays strongly
    everywhere, so head 1 runs in segments."""
    x = _inputs("bf16", 128, 6000, seed=5650, N=1, H=2)
    x["av"][:, 1024:5120, 0, :] -= 8.0
    _check(x, "bf16")


def test_vec_unnormalised_keys_lengthen_the_warm_up():
    """|k| = 2: each token's erase factor I - beta k k^T can stretch the state by
    |1 - 4 beta|, which the warm-up bound includes."""
    x = _inputs("bf16", 128, 2500, seed=5700, N=1, H=2)
    x["k"] = (2.0 * x["k"].float()).to(torch.bfloat16)
    _check(x, "bf16")


def test_vec_packed_long_and_short_sequences():
    x = _inputs("bf16", 128, 6000, seed=5800, N=1, H=2, varlen=True)
    x["cu_seqlens"] = torch.tensor([0, 7, 7, 2100, 2116, 6000], dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(5801)
    x["h0"] = (0.05 * torch.randn((5, 2, 128, 128), generator=g)).cuda()
    _check(x, "bf16")


@pytest.mark.parametrize("which", ["out", "q", "av"])
def test_vec_unaligned_pointer_takes_the_cuda_core_kernels(which):
    """bf16 d = 128 with `out`, or an input, not 16-byte aligned: the fused kernel
    reads and writes 16-byte pieces, so the call runs the CUDA-core kernels; the
    result is the same."""
    x = _inputs("bf16", 128, 40, seed=5900, N=1, H=2)

    def shifted(t):   # a copy of t that starts 2 bytes past an aligned address
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
        u = buf[1:1 + t.numel()].view(t.shape)
        u.copy_(t)
        return u

    out = torch.empty_like(x["v"])
    if which == "out":
        out = shifted(out)
    else:
        x[which] = shifted(x[which])
    hT = torch.empty((1, 2, 128, 128), dtype=torch.float32, device="cuda")
    rc = gdr.gdr_chunk_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], x["h0"], out, hT, None,
                               1, 40, 2, 128, 128, 16, 2.0, gdr.GDR_BF16)
    assert rc == gdr.GDR_OK
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    ro, rh = oracle.oracle_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"], b=2.0)
    assert_close(to64(out), ro, "bf16", "out")
    assert_close(to64(hT), rh, "bf16", "hT")


@pytest.mark.parametrize("case", ["segments", "weak_decay", "packed"])
def test_vec_mma_sync_kernel_still_matches_the_oracle(case, monkeypatch):
    """GDR_VEC_MMA=1 runs the earlier per-channel kernel (mma.sync, the state in
    registers) instead of the tcgen05 one; it stays correct on the shapes that
    exercise its segments, its unsegmented fallback and packed sequences."""
    monkeypatch.setenv("GDR_VEC_MMA", "1")
    if case == "segments":
        x = _inputs("bf16", 128, 3000, seed=5950, N=1, H=2)
    elif case == "weak_decay":
        x = _inputs("bf16", 128, 2000, seed=5951, N=1, H=2, a_mean=-6.0)
    else:
        x = _inputs("bf16", 128, 3000, seed=5952, N=3, H=2, varlen=True)
    _check(x, "bf16")


def test_vec_tensor_core_kernels_agree():
    """The tcgen05 kernel and the mma.sync kernel on the same inputs agree within the
    bf16 tolerance of each against the oracle (both are checked there too)."""
    import os
    x = _inputs("bf16", 128, 2500, seed=5960, N=2, H=3)
    out_tc, hT_tc = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"], b=2.0)
    os.environ["GDR_VEC_MMA"] = "1"
    try:
        out_ms, hT_ms = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], x["av"], x["beta"], h0=x["h0"], b=2.0)
    finally:
        del os.environ["GDR_VEC_MMA"]
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    assert_close(to64(out_tc), to64(out_ms), "bf16", "out, tcgen05 vs mma.sync")
    assert_close(to64(hT_tc), to64(hT_ms), "bf16", "hT, tcgen05 vs mma.sync")
