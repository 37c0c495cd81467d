"""Runs in a process that preloads the AddressSanitizer / UndefinedBehaviorSanitizer
runtimes (tests/test_sanitizers_cpu.py starts it): the oracle's C code, built with both
sanitizers, on small cases of every entry point (compared with the regular build), and
the CUDA library's host code, built with both sanitizers, on the argument refusals that
run without a GPU.  Any sanitizer report aborts the process with a non-zero status.

usage: python sanitized_checks.py <sanitized libgdr_oracle.so> <sanitized librouter_oracle.so>
(GDR_LIB names the sanitized CUDA library.)"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def _case(rng, B, T, H, dk, dv, per_channel=False):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    a = rng.standard_normal((B, T, H, dk) if per_channel else (B, T, H))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, a, beta


def _same(x, y, what):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    assert x.shape == y.shape, what
    assert np.allclose(x, y, rtol=1e-12, atol=1e-12), what


def oracle_cases(lib, rlib):
    rng = np.random.default_rng(7)
    # dense and packed forward, both gates, with and without h0
    q, k, v, a, beta = _case(rng, 2, 37, 3, 8, 6)
    h0 = 0.1 * rng.standard_normal((2, 3, 8, 6))
    for gate in ("bounded", "softplus"):
        for hh in (None, h0):
            r1 = oracle.oracle_fwd(q, k, v, a, beta, h0=hh, gate=gate, _lib_path=lib)
            r0 = oracle.oracle_fwd(q, k, v, a, beta, h0=hh, gate=gate)
            _same(r1[0], r0[0], "fwd out")
            _same(r1[1], r0[1], "fwd hT")
    cu = np.array([0, 0, 5, 21, 21, 40], dtype=np.int64)
    qp, kp, vp, ap, bp = _case(rng, 1, 40, 2, 8, 8)
    h0p = 0.1 * rng.standard_normal((5, 2, 8, 8))
    r1 = oracle.oracle_fwd(qp, kp, vp, ap, bp, h0=h0p, cu_seqlens=cu, _lib_path=lib)
    r0 = oracle.oracle_fwd(qp, kp, vp, ap, bp, h0=h0p, cu_seqlens=cu)
    _same(r1[0], r0[0], "varlen out")
    _same(r1[1], r0[1], "varlen hT")
    # per-channel forward and both backwards
    qc, kc, vc, ac, bc = _case(rng, 1, 29, 2, 8, 6, per_channel=True)
    r1 = oracle.oracle_fwd_vec(qc, kc, vc, ac, bc, _lib_path=lib)
    r0 = oracle.oracle_fwd_vec(qc, kc, vc, ac, bc)
    _same(r1[0], r0[0], "vec out")
    dout = rng.standard_normal(v.shape)
    dhT = 0.1 * rng.standard_normal(h0.shape)
    g1 = oracle.oracle_bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0, _lib_path=lib)
    g0 = oracle.oracle_bwd(q, k, v, a, beta, dout=dout, dhT=dhT, h0=h0)
    for n in g0:
        _same(g1[n], g0[n], "bwd " + n)
    doutc = rng.standard_normal(vc.shape)
    g1 = oracle.oracle_bwd_vec(qc, kc, vc, ac, bc, dout=doutc, _lib_path=lib)
    g0 = oracle.oracle_bwd_vec(qc, kc, vc, ac, bc, dout=doutc)
    for n in g0:
        _same(g1[n], g0[n], "bwd_vec " + n)
    # router: top-k with ties and a load update
    logits = np.round(rng.standard_normal((50, 70)) * 2) / 2
    bias = np.zeros(70, dtype=np.float32)
    t1 = oracle.router_topk(logits.astype(np.float32), bias, 4, _lib_path=rlib)
    t0 = oracle.router_topk(logits.astype(np.float32), bias, 4)
    for x1, x0 in zip(t1, t0):
        assert np.array_equal(np.asarray(x1), np.asarray(x0)), "router topk"
    u1 = oracle.router_update(t0[2], bias, mode="proportional", _lib_path=rlib)
    u0 = oracle.router_update(t0[2], bias, mode="proportional")
    assert np.array_equal(u1[0], u0[0]), "router update"


def library_refusals():
    import chunked_gated_delta_07_gb300 as gdr
    assert os.environ.get("GDR_LIB") == gdr.LIB_PATH
    lib = gdr.lib()
    for code in range(9):
        assert gdr.gdr_status_string(code)
    p = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20]

    def fwd(**kw):
        base = dict(q=p[0], k=p[1], v=p[2], a=p[3], beta=p[4], h0=None, out=6 << 20, hT=None,
                    cu_seqlens=None, B=1, T=64, H=2, dk=128, dv=128, chunk=16, b=2.0,
                    dtype=gdr.GDR_BF16, gate=gdr.GDR_GATE_BOUNDED, path=gdr.GDR_PATH_AUTO,
                    workspace=None, workspace_bytes=0, stream=0)
        base.update(kw)
        return gdr.gdr_chunk_fwd_ex(**base)

    cases = [dict(B=0), dict(H=0), dict(T=-1), dict(dk=96), dict(chunk=8), dict(b=float("nan")),
             dict(q=None), dict(out=1 << 20), dict(hT=(5 << 20) + 8), dict(h0=7 << 20, hT=(7 << 20) + 4),
             dict(T=1 << 41), dict(path=9), dict(dtype=7)]
    for kw in cases:
        assert fwd(**kw) != gdr.GDR_OK, kw
    far = dict(q=1 << 52, k=2 << 52, v=3 << 52, a=4 << 52, beta=5 << 52, out=6 << 52)
    for kw in (dict(far, T=1 << 20, H=16), dict(far, T=1 << 40, H=1 << 22)):
        args = dict(h0=None, hT=None, B=1, T=64, H=2, dk=128, dv=128, chunk=16, b=2.0,
                    dtype=gdr.GDR_BF16, gate=gdr.GDR_GATE_BOUNDED, stream=0)
        args.update(kw)
        assert gdr.gdr_chunk_fwd_noalloc(args["q"], args["k"], args["v"], args["a"], args["beta"],
                                         None, args["out"], None, args["B"], args["T"], args["H"], 128, 128,
                                         16, 2.0, gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED, 0) != gdr.GDR_OK
    for args in ((2, 4096, 16, 128, 128, 16, gdr.GDR_BF16, gdr.GDR_PATH_TC),
                 (1, 0, 1, 64, 64, 64, gdr.GDR_F32, gdr.GDR_PATH_SIMT),
                 (0, 4096, 16, 128, 128, 16, gdr.GDR_BF16, gdr.GDR_PATH_AUTO)):
        gdr.gdr_chunk_fwd_workspace_size(*args)
    assert gdr.gdr_recurrent_fwd(*p, (7 << 20) + 4, 6 << 20, 1, 1, 2, 128, 128, 2.0, gdr.GDR_BF16,
                                 gdr.GDR_GATE_BOUNDED, 0) == gdr.GDR_ERR_INVALID_ARG
    assert lib is not None


if __name__ == "__main__":
    if len(sys.argv) > 3 and sys.argv[3] == "--forward-only":   # the planted-fault run
        rng = np.random.default_rng(7)
        q, k, v, a, beta = _case(rng, 1, 9, 1, 8, 6)
        oracle.oracle_fwd(q, k, v, a, beta, _lib_path=sys.argv[1])
        print("sanitized checks: ok")
        sys.exit(0)
    oracle_cases(sys.argv[1], sys.argv[2])
    library_refusals()
    print("sanitized checks: ok")
