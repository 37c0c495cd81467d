"""Full-size parity of the backward, per-channel decay and router rows: the
workloads the benchmark times, at their sizes and in its launch configuration,
checked against the CPU oracles on outputs they can compute in seconds.

* backward, 8 sequences x 4096 tokens x 16 heads (bf16, d = 128): every gradient
  of two sampled (sequence, head) pairs, the oracle run on those pairs alone
  (heads are independent).
* per-channel decay, the packed 1M-token batch: every output and final state of
  one sampled head of two sampled sequences (one long, one short).
* router, a 1M-token window over 896 experts, k = 8: the picked experts of 4096
  sampled tokens against the oracle on those rows (bit for bit), and the counts
  against the histogram of all picked experts.
Tolerances as in the small parity tests.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle
from gdr_inputs import WORKLOADS, make_channel_gate, make_inputs, make_router_logits
from gpu_helpers import assert_close, rel_l2, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_07_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)


def test_backward_full_size_sampled_pairs():
    N, T, H, d = 8, 4096, 16, 128
    x = make_inputs(WORKLOADS["t1m"].with_(B=N, h0_std=0.02, seed=4500), device="cuda", T=T)
    g = torch.Generator(device="cuda").manual_seed(4501)
    dout = torch.randn(x["v"].shape, generator=g, device="cuda").to(torch.bfloat16)
    dhT = 0.1 * torch.randn((N, H, d, d), generator=g, device="cuda")
    got = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], dout=dout, dhT=dhT,
                        h0=x["h0"], b=2.0)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    names = ("dq", "dk", "dv", "da", "dbeta", "dh0")
    for n, h in ((3, 5), (7, 14)):
        sl = lambda t: t[n:n + 1, :, h:h + 1].contiguous().cpu()
        ref = oracle.oracle_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["a"]), sl(x["beta"]),
                                dout=sl(dout), dhT=dhT[n:n + 1, h:h + 1].cpu(),
                                h0=x["h0"][n:n + 1, h:h + 1].cpu(), b=2.0)
        for name, t in zip(names, got):
            mine = to64(t[n:n + 1, h:h + 1] if name == "dh0" else t[n:n + 1, :, h:h + 1])
            r = ref[name]
            rl = rel_l2(mine, r)
            lim = 5e-2 * max(1.0, float(np.abs(r).max()))
            assert rl <= 1e-2, f"({n},{h}) {name}: rel-L2 {rl:.3e}"
            assert float(np.abs(mine - r).max()) <= lim, f"({n},{h}) {name}: max-abs"


def test_vec_full_size_sampled_sequences():
    w = WORKLOADS["varlen_1m"]
    x = make_inputs(w, device="cuda")
    av = make_channel_gate(x, w.seed + 7)
    out, hT = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"],
                                cu_seqlens=x["cu_seqlens"], b=w.b)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    cu = x["cu_seqlens"].cpu().numpy()
    lens = np.diff(cu)
    long_seq = int(np.argsort(lens)[len(lens) // 2])   # a median-length sequence
    short_seq = int(np.argmin(lens))
    for n, h in ((long_seq, 6), (short_seq, 11)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[:, t0:t1, h:h + 1].contiguous().cpu()
        ro, rh = oracle.oracle_fwd_vec(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(av), sl(x["beta"]),
                                       h0=x["h0"][n:n + 1, h:h + 1].cpu(), b=w.b)
        assert_close(to64(out[:, t0:t1, h:h + 1]), ro, "bf16", f"seq {n} head {h} out")
        assert_close(to64(hT[n:n + 1, h:h + 1]), rh, "bf16", f"seq {n} head {h} hT")


def test_router_full_window_sampled_tokens():
    T, E, k = 1 << 20, 896, 8
    x, bias = make_router_logits(T, E, 6000, "bf16", device="cuda")
    load = torch.zeros(E, dtype=torch.int64, device="cuda")
    idx, sel = gdr.router_topk(x, bias, k, load=load)
    torch.cuda.synchronize()
    assert gdr.gdr_get_status() == gdr.GDR_OK
    rows = torch.randperm(T, generator=torch.Generator().manual_seed(6001))[:4096].sort().values
    r_idx, r_sel, _ = oracle.router_topk(x[rows.cuda()].cpu(), bias.cpu(), k)
    np.testing.assert_array_equal(idx[rows.cuda()].cpu().numpy(), r_idx)
    np.testing.assert_array_equal(sel[rows.cuda()].cpu().numpy(), r_sel)
    hist = torch.bincount(idx.flatten().long(), minlength=E)
    assert torch.equal(hist, load)
    # every row holds k distinct experts
    s = idx.sort(dim=1).values
    assert bool((s[:, 1:] != s[:, :-1]).all())
