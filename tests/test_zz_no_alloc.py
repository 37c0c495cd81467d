"""gdr_chunk_fwd_noalloc against the regular entry point and the oracle (GPU).

The no-allocation entry point serves callers that may not allocate device
memory when they run the pass (graph capture, engines that pre-reserve all
device memory, allocation-free loops).  It keeps its scratch in a static
device array shared by every call, so this test calls it twice in a row on
different inputs and checks each result against gdr_chunk_fwd_ex (CUDA-core
path, ordinary workspace) and against the fp64 oracle, within the parity
tolerance of the other tests; a zero-token call must leave hT = h0.  The
argument refusals (no launch) are covered on the CPU in test_abi_cpu.py.
The file is named so pytest collects it last.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, run_oracle, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _regular(x, dcode, gcode):
    out = torch.empty_like(x["v"])
    hT = torch.empty((x["B"], x["H"], x["dk"], x["dv"]), dtype=torch.float32, device="cuda")
    rc = gdr.gdr_chunk_fwd_ex(x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], out, hT, None,
                              x["B"], x["T"], x["H"], x["dk"], x["dv"], x["chunk"], x["b"], dcode,
                              gcode, gdr.GDR_PATH_SIMT, None, 0, None)
    assert rc == gdr.GDR_OK
    return out, hT


def _noalloc(x, dcode, gcode):
    out = torch.empty_like(x["v"])
    hT = torch.full((x["B"], x["H"], x["dk"], x["dv"]), float("nan"), dtype=torch.float32,
                    device="cuda")
    rc = gdr.gdr_chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], out, hT,
                                   x["B"], x["T"], x["H"], x["dk"], x["dv"], x["chunk"], x["b"],
                                   dcode, gcode, None)
    assert rc == gdr.GDR_OK
    return out, hT


CASES = [
    (WORKLOADS["b2_t4k"].with_(H=4, seed=71), 300, "bf16", gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED),
    (WORKLOADS["small_fp32"].with_(seed=72, h0_std=0.1, gate="softplus", a_std=3.0), 201, "f32",
     gdr.GDR_F32, gdr.GDR_GATE_SOFTPLUS),
]


def test_noalloc_matches_regular_and_oracle_on_two_calls_in_a_row():
    for w, T, tol, dcode, gcode in CASES:
        x = make_inputs(w, device="cuda", T=T)
        o_n, h_n = _noalloc(x, dcode, gcode)
        torch.cuda.synchronize()
        assert gdr.gdr_get_status() == gdr.GDR_OK
        o_r, h_r = _regular(x, dcode, gcode)
        torch.cuda.synchronize()
        assert_close(to64(o_n), to64(o_r), tol, "out vs regular")
        assert_close(to64(h_n), to64(h_r), tol, "hT vs regular")
        ref_o, ref_h = run_oracle(x)
        assert_close(to64(o_n), ref_o.reshape(o_n.shape), tol, "out vs oracle")
        assert_close(to64(h_n), ref_h.reshape(h_n.shape), tol, "hT vs oracle")


def test_noalloc_zero_tokens_copies_the_entering_state():
    w = WORKLOADS["b2_t4k"].with_(H=3, seed=73)
    x = make_inputs(w, device="cuda", T=16)
    x = dict(x, T=0, **{n: x[n][:, :0].contiguous() for n in ("q", "k", "v", "a", "beta")})
    o_n, h_n = _noalloc(x, gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED)
    torch.cuda.synchronize()
    assert o_n.numel() == 0
    np.testing.assert_array_equal(h_n.cpu().numpy(), x["h0"].cpu().numpy())
