"""Runs small parity cases of the forward and backward passes on the checking build of the library
(device-side index checks, GDR_DEBUG), named by GDR_LIB: every case must match the
oracle at the usual tolerances and leave the status word clean (no check failed).
Started by tests/test_debug_build_gpu.py in a process of its own."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import chunked_gated_delta_07_gb300 as gdr  # noqa: E402
from gdr_inputs import WORKLOADS, make_inputs, softplus_variant  # noqa: E402
from gpu_helpers import assert_close, run_oracle, to64  # noqa: E402


def run(x, path, **kw):
    out, hT = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"],
                            cu_seqlens=x["cu_seqlens"], chunk=kw.get("chunk", x["chunk"]), b=x["b"],
                            gate=x["gate"], path=path)
    st = gdr.gdr_get_status()
    assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
    return out, hT


def main():
    assert os.environ.get("GDR_LIB") == gdr.LIB_PATH and "debug" in gdr.LIB_PATH
    torch.cuda.set_device(0)
    cases = [
        (WORKLOADS["b2_t4k"].with_(H=3, seed=1030), 1000, ("simt", "tc"), "bf16"),
        (WORKLOADS["small_fp32"].with_(seed=1031, h0_std=0.1), 201, ("simt",), "f32"),
        (WORKLOADS["varlen_1m"].with_(len_min=30, len_max=700, seed=1032), 2500, ("simt", "tc"), "bf16"),
        (softplus_variant(WORKLOADS["varlen_1m"].with_(len_min=30, len_max=900, seed=1033)), 3000,
         ("tc",), "bf16"),
    ]
    os.environ["GDR_TC_SEG_CHUNKS"] = "3"   # many segments: transition, combine and output passes
    for w, T, paths, tol in cases:
        x = make_inputs(w, device="cuda", T=T)
        ro, rh = run_oracle(x)
        for path in paths:
            out, hT = run(x, path)
            assert_close(to64(out), ro.reshape(out.shape), tol, f"{w.name} out [{path}]")
            assert_close(to64(hT), rh.reshape(hT.shape), tol, f"{w.name} hT [{path}]")
    # the per-channel decay forward (tcgen05 kernel): segments with warm-up tiles, packed
    # sequences with a ragged end
    import oracle
    from gdr_inputs import make_channel_gate
    for w, T in [(WORKLOADS["b2_t4k"].with_(B=1, H=2, seed=1035, h0_std=0.05), 3000),
                 (WORKLOADS["varlen_1m"].with_(H=2, len_min=30, len_max=1500, seed=1036), 3001)]:
        x = make_inputs(w, device="cuda", T=T)
        av = make_channel_gate(x, 1037)
        out, hT = gdr.chunk_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"],
                                    cu_seqlens=x["cu_seqlens"], b=w.b)
        st = gdr.gdr_get_status()
        assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
        cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
        ro, rh = oracle.oracle_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], h0=x["h0"], cu_seqlens=cu,
                                       b=w.b)
        assert_close(to64(out), ro, "bf16", f"{w.name} per-channel out")
        assert_close(to64(hT), rh, "bf16", f"{w.name} per-channel hT")
    # the chunked backward (the two tcgen05 state chains and the per-tile kernel):
    # 64-tile segments with warm-up tiles and a ragged end, one decay per token or per
    # key channel
    from gpu_helpers import rel_l2
    for per_channel in (False, True):
        w = WORKLOADS["b2_t4k"].with_(B=1, H=2, seed=1038, h0_std=0.05)
        x = make_inputs(w, device="cuda", T=2503)
        g = torch.Generator(device="cpu").manual_seed(1039)
        dout = torch.randn(x["v"].shape, generator=g).to(torch.bfloat16).cuda()
        dhT = (0.1 * torch.randn((1, 2, 128, 128), generator=g)).cuda()
        a = make_channel_gate(x, 1040) if per_channel else x["a"]
        fn = gdr.chunk_bwd_vec if per_channel else gdr.chunk_bwd
        ofn = oracle.oracle_bwd_vec if per_channel else oracle.oracle_bwd
        got = fn(x["q"], x["k"], x["v"], a, x["beta"], dout=dout, dhT=dhT, h0=x["h0"], b=w.b)
        st = gdr.gdr_get_status()
        assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
        ref = ofn(x["q"], x["k"], x["v"], a, x["beta"], dout=dout, dhT=dhT, h0=x["h0"], b=w.b)
        for name, gv in zip(("dq", "dk", "dv", "da", "dbeta", "dh0"), got):
            rl = rel_l2(to64(gv), ref[name])
            assert rl <= 1e-2, f"backward (per channel: {per_channel}) {name}: rel-L2 {rl:.3e}"
    # zero tokens
    x = make_inputs(WORKLOADS["b2_t4k"].with_(H=2, seed=1034), device="cuda", T=0)
    for path in ("simt", "tc"):
        _, hT = run(x, path)
        assert torch.equal(hT, x["h0"])
    print("checking build: ok")


if __name__ == "__main__":
    main()
