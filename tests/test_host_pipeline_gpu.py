"""The host-buffer entry point on inputs large enough to be pipelined.

Past 2^21 (token, head) units, gdr_chunk_fwd_host cuts the tokens into pieces:
tile-aligned token ranges of every sequence for dense input, with the state
carried from piece to piece; groups of whole sequences for packed input.  It
copies piece p + 1 in and piece p - 1 out while piece p runs.  Its result must
equal the device-buffer entry point's up to the rounding of a different segment
split, within the bf16 tolerance of every other comparison.
"""
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, run_gpu, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _host_call(x, h0):
    host = [x[n].cpu().pin_memory() for n in ("q", "k", "v", "a", "beta")]
    hh0 = None if h0 is None else h0.cpu().pin_memory()
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu()
    out = torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory()
    hT = torch.empty((x["N"], x["H"], x["dk"], x["dv"]), dtype=torch.float32).pin_memory()
    rc = gdr.gdr_chunk_fwd_host(*host, hh0, out, hT, cu, x["N"], x["T"], x["H"], x["dk"],
                                x["dv"], x["chunk"], x["b"], gdr.GDR_BF16,
                                gdr.GDR_GATE_BOUNDED if x["gate"] == "bounded" else gdr.GDR_GATE_SOFTPLUS,
                                gdr.GDR_PATH_AUTO, None)
    assert rc == gdr.GDR_OK, gdr.gdr_status_string(rc)
    return out, hT


@pytest.mark.parametrize("B,T", [(1, 262144 + 37), (2, 131072 + 5)])
def test_dense_pieces_carry_the_state(B, T):
    w = WORKLOADS["b2_t4k"].with_(B=B, H=8, h0_std=0.02, seed=2101 + B)
    x = make_inputs(w, device="cuda", T=T)
    assert x["T"] * B * x["H"] >= 1 << 21
    out_d, hT_d = run_gpu(x)
    out_h, hT_h = _host_call(x, x["h0"])
    assert_close(to64(out_h), to64(out_d), "bf16", "out host vs device")
    assert_close(to64(hT_h), to64(hT_d), "bf16", "hT host vs device")


def test_packed_groups_of_sequences():
    w = WORKLOADS["varlen_1m"].with_(H=8, len_min=512, len_max=40000, seed=2110)
    x = make_inputs(w, device="cuda", T=300000)
    assert x["N"] >= 4
    out_d, hT_d = run_gpu(x)
    out_h, hT_h = _host_call(x, x["h0"])
    assert_close(to64(out_h), to64(out_d), "bf16", "out host vs device")
    assert_close(to64(hT_h), to64(hT_d), "bf16", "hT host vs device")
