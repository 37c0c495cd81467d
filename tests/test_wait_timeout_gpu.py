"""Bounded device waits of the tensor-core forward kernels (scalar and per-channel
gate), made to run out (GPU).

Every wait in tc_chunk_kernel gives up after a limit (2 s), records
GDR_ERR_TIMEOUT in the status word and unwinds: the CTA drains its tile copies
and tensor-core operations and frees its tensor memory before it returns.  The
test hook GDR_TC_WAIT_NS shortens the pipeline waits' limit so that they run
out on a small case (0: every wait looks once, without suspending, so the first
one not already satisfied gives up); the call must return, report the timeout, and leave the
device usable: the next call at the default limit matches the oracle (it could
not allocate tensor memory, or would read stale tiles, if the unwind had leaked
either).  No fault, trap or endless loop is involved.
"""
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, run_gpu, run_oracle, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _tc_available():
    return gdr.gdr_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 16, gdr.GDR_BF16,
                                            gdr.GDR_PATH_TC) > 0


@pytest.mark.parametrize("limit_ns", [0, 1500, 20000])
def test_waits_that_run_out_report_a_timeout_and_unwind(monkeypatch, limit_ns):
    if not _tc_available():
        pytest.skip("tensor-core path unavailable")
    w = WORKLOADS["b2_t4k"].with_(H=3, seed=1020)
    x = make_inputs(w, device="cuda", T=600)
    assert gdr.gdr_get_status() == gdr.GDR_OK
    monkeypatch.setenv("GDR_TC_WAIT_NS", str(limit_ns))
    monkeypatch.setenv("GDR_TC_SEG_CHUNKS", "8")   # transitions, combine and output passes
    gdr.chunk_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"], chunk=16, b=w.b,
                  path="tc")
    st = gdr.gdr_get_status()   # synchronises: the call has returned
    if limit_ns == 0:
        assert st == gdr.GDR_ERR_TIMEOUT, gdr.gdr_status_string(st)
    else:   # a longer limit may or may not run out, depending on where the waits fall
        assert st in (gdr.GDR_OK, gdr.GDR_ERR_TIMEOUT), gdr.gdr_status_string(st)
    monkeypatch.delenv("GDR_TC_WAIT_NS")
    ro, rh = run_oracle(x)
    for _ in range(2):
        out, hT = run_gpu(x, path="tc")   # asserts a clean status
        assert_close(to64(out), ro, "bf16", "out")
        assert_close(to64(hT), rh, "bf16", "hT")


@pytest.mark.parametrize("limit_ns", [0, 1500])
def test_per_channel_kernel_waits_that_run_out_unwind(monkeypatch, limit_ns):
    """The same for the per-channel tcgen05 kernel (gdr_chunk_fwd_vec, bf16 d = 128),
    with segments and warm-up tiles: the timed-out call reports GDR_ERR_TIMEOUT (limit
    0), and the next two calls match the oracle."""
    import oracle
    from gdr_inputs import make_channel_gate
    w = WORKLOADS["b2_t4k"].with_(B=1, H=2, seed=1025, h0_std=0.05)
    x = make_inputs(w, device="cuda", T=2000)
    av = make_channel_gate(x, 1026)
    assert gdr.gdr_get_status() == gdr.GDR_OK
    monkeypatch.setenv("GDR_TC_WAIT_NS", str(limit_ns))
    gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"], b=w.b)
    st = gdr.gdr_get_status()
    if limit_ns == 0:
        assert st == gdr.GDR_ERR_TIMEOUT, gdr.gdr_status_string(st)
    else:
        assert st in (gdr.GDR_OK, gdr.GDR_ERR_TIMEOUT), gdr.gdr_status_string(st)
    monkeypatch.delenv("GDR_TC_WAIT_NS")
    ro, rh = oracle.oracle_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"], b=w.b)
    for _ in range(2):
        out, hT = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"], b=w.b)
        torch.cuda.synchronize()
        assert gdr.gdr_get_status() == gdr.GDR_OK
        assert_close(to64(out), ro, "bf16", "out")
        assert_close(to64(hT), rh, "bf16", "hT")


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("limit_ns", [0, 1500])
def test_backward_chain_waits_that_run_out_unwind(monkeypatch, limit_ns, per_channel):
    """The same for the backward's two tcgen05 state chains (tc_fwd_chain_kernel and
    tc_adj_kernel, bf16 d = 128, segments with warm-up tiles): the timed-out call
    reports GDR_ERR_TIMEOUT (limit 0), and the next two calls match the oracle."""
    import numpy as np
    import oracle
    from gdr_inputs import make_channel_gate
    from gpu_helpers import rel_l2
    w = WORKLOADS["b2_t4k"].with_(B=1, H=2, seed=1030, h0_std=0.05)
    x = make_inputs(w, device="cuda", T=2000)
    g = torch.Generator(device="cpu").manual_seed(1031)
    dout = torch.randn(x["v"].shape, generator=g).to(torch.bfloat16).cuda()
    dhT = (0.1 * torch.randn((1, 2, 128, 128), generator=g)).cuda()
    a = make_channel_gate(x, 1032) if per_channel else x["a"]
    fn = gdr.chunk_bwd_vec if per_channel else gdr.chunk_bwd
    ofn = oracle.oracle_bwd_vec if per_channel else oracle.oracle_bwd

    def call():
        return fn(x["q"], x["k"], x["v"], a, x["beta"], dout=dout, dhT=dhT, h0=x["h0"], b=w.b)

    assert gdr.gdr_get_status() == gdr.GDR_OK
    monkeypatch.setenv("GDR_TC_WAIT_NS", str(limit_ns))
    call()
    st = gdr.gdr_get_status()
    if limit_ns == 0:
        assert st == gdr.GDR_ERR_TIMEOUT, gdr.gdr_status_string(st)
    else:
        assert st in (gdr.GDR_OK, gdr.GDR_ERR_TIMEOUT), gdr.gdr_status_string(st)
    monkeypatch.delenv("GDR_TC_WAIT_NS")
    ref = ofn(x["q"], x["k"], x["v"], a, x["beta"], dout=dout, dhT=dhT, h0=x["h0"], b=w.b)
    for _ in range(2):
        got = call()
        torch.cuda.synchronize()
        assert gdr.gdr_get_status() == gdr.GDR_OK
        for name, gv in zip(("dq", "dk", "dv", "da", "dbeta", "dh0"), got):
            r = ref[name]
            assert rel_l2(to64(gv), r) <= 1e-2, name
            lim = 5e-2 * max(1.0, float(np.abs(r).max()))
            assert float(np.abs(to64(gv) - r).max()) <= lim, name
