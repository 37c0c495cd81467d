"""GPU invariants that hold at any size: chaining, tile-size independence,
varlen == separate calls, column independence, determinism."""
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, rel_l2, run_gpu, to64

pytestmark = pytest.mark.gpu


def _paths():
    ps = ["simt"]
    if gdr.gdr_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 16, gdr.GDR_BF16, gdr.GDR_PATH_TC) > 0:
        ps.append("tc")
    return ps


def _slice(x, s, e):
    y = dict(x)
    for n in ("q", "k", "v", "a", "beta"):
        y[n] = x[n][:, s:e].contiguous()
    y["T"] = e - s
    return y


@pytest.mark.parametrize("path", _paths())
def test_chaining(path):
    x = make_inputs(WORKLOADS["b2_t4k"].with_(H=4), device="cuda", T=1000)
    out, hT = run_gpu(x, path=path)
    s = 368   # tile-aligned split
    o1, h1 = run_gpu(_slice(x, 0, s), path=path)
    o2, h2 = run_gpu(_slice(x, s, 1000), path=path, h0=h1)
    # identical tiling on both sides of the split: equal up to the bf16 rounding of out
    assert_close(to64(torch.cat([o1, o2], 1)), to64(out), "bf16", "out")
    if path == "simt":   # same tiles, same fp32 operations on both sides of the split
        assert rel_l2(to64(h2), to64(hT)) < 1e-5
    else:
        # the tensor-core path's segments move with the split, which changes only the
        # rounding (bf16 operands of the tile products): measured 2.3e-3 on out and hT
        assert rel_l2(to64(torch.cat([o1, o2], 1)), to64(out)) < 3e-3
        assert rel_l2(to64(h2), to64(hT)) < 3e-3


@pytest.mark.parametrize("path", _paths())
def test_chunk_size_independence(path):
    x = make_inputs(WORKLOADS["b2_t4k"].with_(H=4), device="cuda", T=777)
    ref_o, ref_h = run_gpu(x, path=path, chunk=16)
    for c in (32, 64):
        tc_ok = gdr.gdr_chunk_fwd_workspace_size(1, 64, 1, 128, 128, c, gdr.GDR_BF16,
                                                 gdr.GDR_PATH_TC) > 0
        o, h = run_gpu(x, path=path if (path == "simt" or tc_ok) else "simt", chunk=c)
        assert_close(to64(o), to64(ref_o), "bf16", f"out c={c}")
        assert_close(to64(h), to64(ref_h), "bf16", f"hT c={c}")


@pytest.mark.parametrize("path", _paths())
def test_varlen_equals_separate_calls(path):
    x = make_inputs(WORKLOADS["varlen_1m"].with_(len_min=50, len_max=900), device="cuda", T=3000)
    out, hT = run_gpu(x, path=path)
    cu = x["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        y = _slice(x, cu[n], cu[n + 1])
        y.update(cu_seqlens=None, B=1, N=1, h0=x["h0"][n:n + 1])
        o, h = run_gpu(y, path=path)
        if path == "simt":   # the same tiles and fp32 operations either way
            assert rel_l2(to64(o), to64(out[:, cu[n]:cu[n + 1]])) < 1e-5
            assert rel_l2(to64(h), to64(hT[n:n + 1])) < 1e-5
        else:
            # the tensor-core path cuts packed and single sequences into segments
            # differently, which changes only the rounding (as in test_chaining)
            assert rel_l2(to64(o), to64(out[:, cu[n]:cu[n + 1]])) < 3e-3
            assert rel_l2(to64(h), to64(hT[n:n + 1])) < 3e-3


@pytest.mark.parametrize("path", _paths())
def test_determinism(path):
    x = make_inputs(WORKLOADS["b2_t4k"].with_(H=4), device="cuda", T=900)
    o1, h1 = run_gpu(x, path=path)
    o2, h2 = run_gpu(x, path=path)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_value_columns_are_independent():
    """Columns of the state evolve independently: zeroing v's second half
    leaves out[..., :64] and hT[..., :64] unchanged (bitwise on the SIMT path,
    whose column split is 32 wide)."""
    x = make_inputs(WORKLOADS["b2_t4k"].with_(H=2), device="cuda", T=500)
    o1, h1 = run_gpu(x, path="simt")
    y = dict(x, v=x["v"].clone(), h0=x["h0"].clone())
    y["v"][..., 64:] = 0
    y["h0"][..., 64:] = 0
    o2, h2 = run_gpu(y, path="simt")
    assert torch.equal(o1[..., :64], o2[..., :64])
    assert torch.equal(h1[..., :64], h2[..., :64])
