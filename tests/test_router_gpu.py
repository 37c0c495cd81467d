"""GPU parity of the quantile-balancing router-bias update (gdr_router_topk and
gdr_router_bias_update) against the CPU oracle: bit-exact.

The selection is an integer decision taken on binary32 scores logit + bias on
both sides, the counts are integers, the quantiles and the bias steps are the
same IEEE operations in the same order ("Deep Dive: The Next Generation of
Ultra-Long Context Sparse MoE LLMs", §4.2; "Core Technologies Behind
Ultra-Long-Context Sparse MoE Large Models", §3.2; "How Trillion-Scale Sparse
MoE Models Achieve Million-Token Long Context Capabilities", §4.3; "Evaluating
Next-Gen Sparse MoE and Long-Context LLMs", §3.2), so every output must match
exactly.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import make_router_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _topk_case(T, E, k, dtype="bf16", ties=False, seed=0, load0=None):
    x, bias = make_router_logits(T, E, seed, dtype, device="cuda", ties=ties)
    if ties:
        bias = torch.zeros_like(bias)
    load = torch.zeros(E, dtype=torch.int64, device="cuda") if load0 is None else load0.clone()
    idx, sel = gdr.router_topk(x, bias, k, load=load)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    r_idx, r_sel, r_load = oracle.router_topk(x, bias, k,
                                              load=None if load0 is None else load0.cpu().numpy())
    np.testing.assert_array_equal(idx.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(sel.cpu().numpy(), r_sel)
    np.testing.assert_array_equal(load.cpu().numpy(), r_load)
    return x, bias, load


@pytest.mark.parametrize("T,E,k", [(1000, 896, 8), (333, 64, 6), (257, 2048, 32), (50, 4, 4),
                                   (100, 1024, 1), (77, 132, 9)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_bit_exact(T, E, k, dtype):
    _topk_case(T, E, k, dtype, seed=T + E + k)


@pytest.mark.parametrize("T,E,k,dtype", [(12000, 132, 9, "bf16"), (12000, 896, 8, "f32"),
                                         (6000, 2048, 32, "f32"), (12000, 512, 4, "bf16")])
def test_topk_bit_exact_many_tokens_per_warp(T, E, k, dtype):
    """Enough tokens that every warp ranks several (one resident wave of blocks, each warp
    walking its tokens with the next row in flight), so the row buffers rotate."""
    _topk_case(T, E, k, dtype, seed=T + 7 * E + k)


@pytest.mark.parametrize("E,k", [(896, 8), (64, 16), (256, 32)])
def test_topk_with_many_ties(E, k):
    """Logits on a half-integer grid and a zero bias: many equal scores, so the
    threshold gathers more than fit and the arg-max rounds decide."""
    _topk_case(400, E, k, "bf16", ties=True, seed=E + k)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_signed_zero_ties(dtype):
    """Scores of -0 and +0 are equal (binary32 comparison): the lower expert index
    goes first, on both sides, whichever zero each score carries."""
    T, E, k = 300, 128, 8
    g = torch.Generator().manual_seed(11)
    vals = torch.tensor([0.0, -0.0, 0.5, -0.5])
    x = vals[torch.randint(0, 4, (T, E), generator=g)]
    x = x.to(torch.bfloat16 if dtype == "bf16" else torch.float32).cuda()
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    bias[::3] = -0.0
    load = torch.zeros(E, dtype=torch.int64, device="cuda")
    idx, sel = gdr.router_topk(x, bias, k, load=load)
    torch.cuda.synchronize()
    r_idx, r_sel, r_load = oracle.router_topk(x, bias, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(load.cpu().numpy(), r_load)


def test_topk_nan_scores_stay_in_bounds():
    """NaN logits give an unspecified selection, but every pick is a distinct valid
    expert of its token and the counts add up to T k."""
    T, E, k = 200, 896, 8
    x, bias = make_router_logits(T, E, 5, "bf16", device="cuda")
    x = x.clone()
    x[::2, ::7] = float("nan")      # some NaN in every other token
    x[1::10, :] = float("nan")      # tokens whose scores are all NaN
    load = torch.zeros(E, dtype=torch.int64, device="cuda")
    idx, _ = gdr.router_topk(x, bias, k, load=load)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    got = idx.cpu().numpy()
    assert got.min() >= 0 and got.max() < E
    assert all(len(set(r)) == k for r in got.tolist())
    assert int(load.sum()) == T * k
    # tokens without NaN are still exact
    clean = np.arange(T)[(np.arange(T) % 2 == 1) & (np.arange(T) % 10 != 1)]
    r_idx, _, _ = oracle.router_topk(x[torch.as_tensor(clean, device=x.device)], bias, k)
    np.testing.assert_array_equal(got[clean], r_idx)


def test_load_accumulates_and_zero_tokens():
    x, bias, load = _topk_case(500, 896, 8, seed=1)
    _topk_case(300, 896, 8, seed=2, load0=load)
    empty = torch.empty((0, 896), dtype=torch.bfloat16, device="cuda")
    before = load.clone()
    idx = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    assert gdr.gdr_router_topk(empty, bias, idx, None, load, 0, 896, 8, gdr.GDR_BF16) == gdr.GDR_OK
    torch.cuda.synchronize()
    assert torch.equal(load, before)


@pytest.mark.parametrize("mode,q_lo,q_hi", [("sign", 0.1, 0.9), ("sign", 0.5, 0.5),
                                            ("proportional", 0.75, 0.75), ("sign", 0.0, 1.0),
                                            ("proportional", 0.3, 0.37)])
@pytest.mark.parametrize("E", [896, 7, 2048])
def test_bias_update_bit_exact(mode, q_lo, q_hi, E):
    g = torch.Generator().manual_seed(E)
    load = torch.randint(0, 100000, (E,), generator=g, dtype=torch.int64)
    load[: E // 3] = load[E // 3]                     # repeated loads
    bias = 0.01 * torch.randn(E, generator=g)
    b_gpu = bias.cuda()
    thr = gdr.router_bias_update(load.cuda(), b_gpu, mode, q_lo, q_hi, 1e-3)
    torch.cuda.synchronize()
    ref_b, ref_thr = oracle.router_update(load.numpy(), bias.numpy(), mode, q_lo, q_hi, 1e-3)
    np.testing.assert_array_equal(b_gpu.cpu().numpy(), ref_b)
    assert tuple(thr.cpu().tolist()) == ref_thr


def test_balancing_loop_reduces_imbalance():
    """Several windows of routing + sign update on skewed logits: the spread of
    the loads shrinks, and every window matches the oracle bit for bit."""
    E, k, T = 128, 4, 4096
    x, bias = make_router_logits(T, E, 77, "bf16", device="cuda", skew=0.5)
    b_cpu = bias.cpu().numpy()
    spreads = []
    for _ in range(8):
        load = torch.zeros(E, dtype=torch.int64, device="cuda")
        gdr.router_topk(x, bias, k, load=load, want_logits=False)
        gdr.router_bias_update(load, bias, "sign", 0.1, 0.9, 0.05)
        torch.cuda.synchronize()
        _, _, r_load = oracle.router_topk(x, b_cpu, k)
        np.testing.assert_array_equal(load.cpu().numpy(), r_load)
        b_cpu, _ = oracle.router_update(r_load, b_cpu, "sign", 0.1, 0.9, 0.05)
        np.testing.assert_array_equal(bias.cpu().numpy(), b_cpu)
        spreads.append(int(r_load.max() - r_load.min()))
    assert spreads[-1] < spreads[0]


def test_bad_args():
    x, bias = make_router_logits(8, 896, 0, "bf16", device="cuda")
    idx = torch.empty((8, 8), dtype=torch.int32, device="cuda")
    load = torch.zeros(896, dtype=torch.int64, device="cuda")
    B = gdr.GDR_BF16
    assert gdr.gdr_router_topk(x, bias, idx, None, load, 8, 896, 33, B) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_router_topk(x, bias, idx, None, load, 8, 894, 8, B) == gdr.GDR_ERR_UNSUPPORTED
    assert gdr.gdr_router_topk(x, bias, idx, None, load, 8, 896, 0, B) == gdr.GDR_ERR_INVALID_ARG
    assert gdr.gdr_router_topk(x.view(-1)[1:], bias, idx, None, load, 7, 896, 8, B) == \
        gdr.GDR_ERR_INVALID_ARG                       # logits not 16-byte aligned
    assert gdr.gdr_router_topk(x, bias, x, None, load, 8, 896, 8, B) == gdr.GDR_ERR_INVALID_ARG
    thr = torch.empty(2, dtype=torch.float64, device="cuda")
    assert gdr.gdr_router_bias_update(load, bias, thr, 896, 0, -0.1, 0.9, 1e-3) == \
        gdr.GDR_ERR_INVALID_ARG
    assert gdr.gdr_router_bias_update(load, bias, thr, 4096, 0, 0.1, 0.9, 1e-3) == \
        gdr.GDR_ERR_UNSUPPORTED
