"""GPU special cases whose answer the mathematics fixes without the oracle.

Each case runs on both kernel families (CUDA-core and tensor-core) through the
C ABI and is compared with a closed form computed here in fp64, and with the
oracle.  The closed forms follow from the recurrence
    H_t = a_t H_{t-1} + beta_t k_t (v_t - a_t H_{t-1}^T k_t)^T,  o_t = H_t^T q_t
("Evaluating Next-Gen Sparse MoE and Long-Context LLMs", §2.2) and the bounded
gate g = -b sigmoid(a) ("Deep Dive: The Next Generation of Ultra-Long Context
Sparse MoE LLMs", §3.3).
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_inputs
from gpu_helpers import assert_close, run_gpu, run_oracle, to64

pytestmark = pytest.mark.gpu


def _tc_available():
    return gdr.gdr_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 16, gdr.GDR_BF16,
                                            gdr.GDR_PATH_TC) > 0


PATHS = ["simt", "tc"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def _need(path):
    if path == "tc" and not _tc_available():
        pytest.skip("tensor-core path unavailable")


def _global_logdecay(x, b):
    """fp64 cumulative log-decay along each sequence, [B, T, H]."""
    a = to64(x["a"])
    g = np.vectorize(lambda z: oracle.gate(z, b, "bounded"))(a)
    return np.cumsum(g, axis=1)


@pytest.mark.parametrize("path", PATHS)
def test_beta_zero_is_pure_decay(path):
    """beta = 0 writes nothing: o_t = e^{G_t} h0^T q_t and hT = e^{G_T} h0, with
    G_t the inclusive cumulative log-decay from the sequence start."""
    _need(path)
    w = WORKLOADS["b2_t4k"].with_(B=1, H=4, a_mean=-6.0, a_std=0.5, h0_std=0.05)
    x = make_inputs(w, device="cuda", T=700)
    x["beta"].zero_()
    out, hT = run_gpu(x, path=path)
    G = _global_logdecay(x, w.b)[0]                      # [T, H]
    h0 = to64(x["h0"])[0]                               # [H, dk, dv]
    q = to64(x["q"])[0]                                 # [T, H, dk]
    ref_out = np.exp(G)[..., None] * np.einsum("thd,hde->the", q, h0)
    ref_hT = np.exp(G[-1])[:, None, None] * h0
    assert_close(to64(out)[0], ref_out, "bf16", "out vs closed form")
    assert_close(to64(hT)[0], ref_hT, "bf16", "hT vs closed form")
    ro, rh = run_oracle(x)
    assert_close(to64(out), ro, "bf16", "out vs oracle")


@pytest.mark.parametrize("path", PATHS)
def test_distinct_basis_keys_reduce_to_gated_linear_attention(path):
    """With keys e_{pi(t)} for a permutation pi (T <= dk) every erase term
    H^T k_t vanishes exactly, so the delta rule is gated linear attention with
    write strength beta:  o_t = sum_{s<=t} e^{G_t - G_s} beta_s (q_t . k_s) v_s."""
    _need(path)
    T, H, d = 128, 2, 128
    w = WORKLOADS["b2_t4k"].with_(B=1, H=H, a_mean=-2.0, h0_std=0.0)
    x = make_inputs(w, device="cuda", T=T)
    gen = torch.Generator().manual_seed(77)
    k = torch.zeros((1, T, H, d))
    for h in range(H):
        perm = torch.randperm(d, generator=gen)[:T]
        k[0, torch.arange(T), h, perm] = 1.0
    x["k"] = k.to(torch.bfloat16).cuda()
    out, hT = run_gpu(x, path=path)
    G = _global_logdecay(x, w.b)[0]                      # [T, H]
    q, kk, v, beta = (to64(x[n])[0] for n in ("q", "k", "v", "beta"))
    ref_out = np.zeros((T, H, d))
    ref_hT = np.zeros((H, d, d))
    for h in range(H):
        dec = np.exp(G[:, None, h] - G[None, :, h]) * np.tri(T)       # [t, s], s <= t
        sc = (q[:, h] @ kk[:, h].T) * dec * beta[None, :, h]
        ref_out[:, h] = sc @ v[:, h]
        wts = np.exp(G[-1, h] - G[:, h]) * beta[:, h]
        ref_hT[h] = (kk[:, h] * wts[:, None]).T @ v[:, h]
    assert_close(to64(out)[0], ref_out, "bf16", "out vs closed form")
    assert_close(to64(hT)[0], ref_hT, "bf16", "hT vs closed form")


@pytest.mark.parametrize("path", PATHS)
def test_overwrite_without_decay(monkeypatch, path):
    """g = 0 (sigmoid(-200) is 0), beta = 1, unit keys and q_t = k_t: each write
    replaces the value stored under its key, so o_t = H_t^T k_t = v_t for every
    t, whatever the earlier keys were.  Keys have four entries of +-1/2, so
    their norm is exactly 1 in bf16.  Short segments make the tensor-core path
    run full (untruncated) transitions, since nothing decays."""
    _need(path)
    monkeypatch.setenv("GDR_TC_SEG_CHUNKS", "8")
    T, H, d = 1200, 2, 128
    w = WORKLOADS["b2_t4k"].with_(B=1, H=H, h0_std=0.0)
    x = make_inputs(w, device="cuda", T=T)
    gen = torch.Generator().manual_seed(78)
    k = torch.zeros((1, T, H, d))
    for t in range(T):
        for h in range(H):
            idx = torch.randperm(d, generator=gen)[:4]
            sign = torch.randint(0, 2, (4,), generator=gen).float() * 2 - 1
            k[0, t, h, idx] = 0.5 * sign
    x["k"] = k.to(torch.bfloat16).cuda()
    x["q"] = x["k"].clone()
    x["a"].fill_(-200.0)
    x["beta"].fill_(1.0)
    out, hT = run_gpu(x, path=path)
    assert_close(to64(out), to64(x["v"]), "bf16", "out vs v")
    ro, rh = run_oracle(x)
    np.testing.assert_allclose(ro, to64(x["v"]), rtol=0, atol=1e-12)   # the oracle is exact here
    assert_close(to64(hT), rh, "bf16", "hT vs oracle")


@pytest.mark.parametrize("path", PATHS)
def test_gate_bound_of_the_pages(path):
    """b = 5, the bound the pages fix, on the 16-head bf16 shape."""
    _need(path)
    w = WORKLOADS["b2_t4k"].with_(b=5.0, a_std=2.0)
    x = make_inputs(w, device="cuda", T=1040)
    out, hT = run_gpu(x, path=path)
    ro, rh = run_oracle(x)
    assert_close(to64(out), ro, "bf16", "out")
    assert_close(to64(hT), rh, "bf16", "hT")
