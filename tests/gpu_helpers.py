"""Shared helpers of the GPU parity tests (runs the C ABI, the oracle, metrics)."""
from __future__ import annotations

import numpy as np
import torch

import chunked_gated_delta_07_gb300 as gdr
import oracle

# tolerances: fp32 workloads rel-L2 <= 1e-4; bf16 workloads rel-L2 <= 1e-2 and
# max-abs <= 5e-2 on both out and hT
TOL = {"f32": dict(rel=1e-4, mabs=None), "bf16": dict(rel=1e-2, mabs=5e-2)}


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return num / den if den > 0 else num


def assert_close(x, ref, dtype, what=""):
    t = TOL[dtype]
    r = rel_l2(x, ref)
    assert r <= t["rel"], f"{what}: rel-L2 {r:.3e} > {t['rel']}"
    if t["mabs"] is not None:
        m = float(np.abs(np.asarray(x, np.float64) - ref).max()) if np.size(ref) else 0.0
        assert m <= t["mabs"], f"{what}: max-abs {m:.3e} > {t['mabs']}"
    return r


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(x, path="auto", chunk=None, h0="input", want_state=True, gate=None, b=None):
    h = x["h0"] if isinstance(h0, str) else h0
    out, hT = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=h,
                            cu_seqlens=x["cu_seqlens"], chunk=chunk or x["chunk"],
                            b=x["b"] if b is None else b, gate=gate or x["gate"], path=path,
                            want_state=want_state)
    torch.cuda.synchronize()
    st = gdr.gdr_get_status()
    assert st == gdr.GDR_OK, gdr.gdr_status_string(st)
    return out, hT


def run_oracle(x, h0="input", gate=None, b=None):
    h = x["h0"] if isinstance(h0, str) else h0
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
    return oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=h, cu_seqlens=cu,
                             b=x["b"] if b is None else b, gate=gate or x["gate"])
