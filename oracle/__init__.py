"""fp64 CPU oracle for the chunked gated delta-rule forward pass.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package; only the tests, the smoke check and the
benchmark's CPU-baseline leg do.  The oracle shares no code with the CUDA
path.

Independent references live here:

* ``oracle_fwd`` -- the token-by-token recurrence in fp64, written in plain C
  (``gdr_oracle.c``, OpenMP over (sequence, head, column block)).  This is the
  definition the chunked GPU method must reproduce.
* ``oracle_fwd_vec`` -- the same recurrence with one decay factor per key
  channel (a is [B,T,H,dk]), pinned by its reduction to ``oracle_fwd`` when all
  channels agree, by the closed form of the per-channel linear-attention sum
  without the erase term, and by exact special cases.
* ``oracle_bwd`` -- the gradients of <dout, out> + <dhT, hT> with respect to
  every input, by the token-by-token adjoint recurrence in fp64 (the same C
  file), pinned by finite differences of ``oracle_fwd``.
* ``router_topk`` / ``router_update`` -- the quantile-balancing router-bias
  update (``router_oracle.c``): top-k of logit + bias per token, per-expert
  load counts, linear-interpolation quantiles and the sign or proportional
  bias step, pinned by numpy's stable argsort and quantile and by closed forms.
* ``chunk_ref`` -- the chunk-parallel (WY / UT) form in fp64 numpy, used only
  to check the GPU's intermediate stages (gate cumsum, W, U) one by one, and the
  chunked backward's per-tile formulas, checked against ``oracle_bwd`` and
  ``oracle_bwd_vec``.

Citation keys used in this package (page title, section):
  P1 = "Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs"
  P2 = "Core Technologies Behind Ultra-Long-Context Sparse MoE Large Models"
  P3 = "How Trillion-Scale Sparse MoE Models Achieve Million-Token Long Context
        Capabilities"
  P4 = "Evaluating Next-Gen Sparse MoE and Long-Context LLMs"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "libgdr_oracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32, F64 = 0, 1, 2
GATES = {"bounded": 0, "softplus": 1}


_RSRC = os.path.join(_HERE, "router_oracle.c")
_RLIB = os.path.join(_HERE, "librouter_oracle.so")
_rlib = None


def _compile(src, lib, force):
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(src):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build_sanitized(out_dir: str, gdr_src: str | None = None) -> tuple[str, str]:
    """Compile both C files with AddressSanitizer and UndefinedBehaviorSanitizer into
    out_dir (for the sanitizer tests, which load them in a process that preloads the
    sanitizer runtimes); ``gdr_src`` replaces gdr_oracle.c (a planted fault).  Returns
    (libgdr_oracle, librouter_oracle) paths."""
    os.makedirs(out_dir, exist_ok=True)
    outs = []
    for src, name in ((gdr_src or _SRC, "libgdr_oracle.so"), (_RSRC, "librouter_oracle.so")):
        lib = os.path.join(out_dir, name)
        cmd = ["gcc", "-O1", "-g", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
               "-fno-omit-frame-pointer", "-o", lib, src, "-lm"]
        subprocess.run(cmd, check=True)
        outs.append(lib)
    return outs[0], outs[1]


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c into libgdr_oracle.so and router_oracle.c into
    librouter_oracle.so next to them (gcc, OpenMP, ISO C11: no FMA contraction)."""
    _compile(_RSRC, _RLIB, force)
    return _compile(_SRC, _LIB, force)


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.gdr_oracle_fwd.restype = ctypes.c_int
    lib.gdr_oracle_fwd.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gdr_oracle_fwd_vec.restype = ctypes.c_int
    lib.gdr_oracle_fwd_vec.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gdr_oracle_bwd.restype = ctypes.c_int
    lib.gdr_oracle_bwd.argtypes = (
        [ctypes.c_void_p] * 5 + [ctypes.c_int] + [ctypes.c_void_p] * 9
        + [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
           ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int])
    lib.gdr_oracle_bwd_vec.restype = ctypes.c_int
    lib.gdr_oracle_bwd_vec.argtypes = lib.gdr_oracle_bwd.argtypes
    lib.gdr_oracle_gate.restype = ctypes.c_double
    lib.gdr_oracle_gate.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_int]
    lib.gdr_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _rbind(path):
    lib = ctypes.CDLL(path)
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.gdr_oracle_router_topk.restype = I
    lib.gdr_oracle_router_topk.argtypes = [P, I, P, I64, I, I, P, P, P]
    lib.gdr_oracle_router_update.restype = I
    lib.gdr_oracle_router_update.argtypes = [P, I, P, I, D, D, ctypes.c_float, P]
    return lib


def _rload():
    global _rlib
    with _lock:
        if _rlib is None:
            build()
            _rlib = _rbind(_RLIB)
    return _rlib


ROUTER_MODES = {"sign": 0, "proportional": 1}


def router_topk(logits, bias, k, load=None, _lib_path=None):
    """Top-k experts of every token by score logit + bias (binary32 add), ties to
    the lower index.  logits [T, E] (bf16 bit patterns or fp32), bias [E] fp32.
    Returns (idx [T, k] int32 in rank order, selected logits [T, k] fp32, load
    [E] int64 = the given load (or zeros) plus this call's counts)."""
    lib = _rload() if _lib_path is None else _rbind(_lib_path)
    xa, dt = _as_array(logits)
    assert dt in (BF16, F32), "logits must be bf16 or fp32"
    T, E = xa.shape
    b = np.ascontiguousarray(np.asarray(bias.cpu().numpy() if hasattr(bias, "cpu") else bias,
                                        dtype=np.float32))
    idx = np.zeros((T, k), dtype=np.int32)
    sel = np.zeros((T, k), dtype=np.float32)
    ld = np.zeros(E, dtype=np.int64) if load is None else np.array(load, dtype=np.int64)
    rc = lib.gdr_oracle_router_topk(xa.ctypes.data, dt, b.ctypes.data, T, E, k, idx.ctypes.data,
                                    sel.ctypes.data, ld.ctypes.data)
    if rc != 0:
        raise ValueError(f"gdr_oracle_router_topk rejected its arguments (code {rc})")
    return idx, sel, ld


def router_update(load, bias, mode="sign", q_lo=0.1, q_hi=0.9, eta=1e-3, _lib_path=None):
    """Quantile-balancing bias update.  Returns (new bias [E] fp32, (Q_lo, Q_hi))."""
    lib = _rload() if _lib_path is None else _rbind(_lib_path)
    ld = np.ascontiguousarray(np.asarray(load, dtype=np.int64))
    b = np.array(bias.cpu().numpy() if hasattr(bias, "cpu") else bias, dtype=np.float32)
    thr = np.zeros(2, dtype=np.float64)
    rc = lib.gdr_oracle_router_update(ld.ctypes.data, ld.shape[0], b.ctypes.data,
                                      ROUTER_MODES[mode], float(q_lo), float(q_hi), float(eta),
                                      thr.ctypes.data)
    if rc != 0:
        raise ValueError(f"gdr_oracle_router_update rejected its arguments (code {rc})")
    return b, (float(thr[0]), float(thr[1]))


def _as_array(x):
    """Return (contiguous numpy array, dtype code) holding x's stored values.

    bf16 torch tensors are passed as their raw 16-bit patterns so that the C
    side widens exactly the values a GPU consumed."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                x = x.cpu()
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16)), BF16
            if x.dtype == torch.float32:
                return np.ascontiguousarray(x.numpy()), F32
            return np.ascontiguousarray(x.to(torch.float64).numpy()), F64
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    return np.ascontiguousarray(x, dtype=np.float64), F64


def oracle_bwd(q, k, v, a, beta, dout=None, dhT=None, h0=None, cu_seqlens=None,
               b: float = 2.0, gate: str = "bounded", nthreads: int = 0,
               _lib_path: str | None = None):
    """fp64 gradients of <dout, out> + <dhT, hT> of the token-by-token forward.

    Same shapes as ``oracle_fwd``; dout is [B,T,H,dv] and dhT [N,H,dk,dv] (None
    means zero).  Returns a dict with dq, dk [B,T,H,dk], dv [B,T,H,dv], da, dbeta
    [B,T,H] and dh0 [N,H,dk,dv], all fp64, with respect to the stored input values
    (bf16 inputs widened exactly)."""
    return _bwd("gdr_oracle_bwd", q, k, v, a, beta, dout, dhT, h0, cu_seqlens, b, gate, nthreads,
                _lib_path)


def oracle_bwd_vec(q, k, v, a, beta, dout=None, dhT=None, h0=None, cu_seqlens=None,
                   b: float = 2.0, gate: str = "bounded", nthreads: int = 0,
                   _lib_path: str | None = None):
    """fp64 gradients of <dout, out> + <dhT, hT> of the per-channel decay forward
    (``oracle_fwd_vec``): a is [B,T,H,dk] and so is the returned da.  It keeps every
    state of a sequence, so it is meant for small cases."""
    return _bwd("gdr_oracle_bwd_vec", q, k, v, a, beta, dout, dhT, h0, cu_seqlens, b, gate,
                nthreads, _lib_path)


def _bwd(fn, q, k, v, a, beta, dout, dhT, h0, cu_seqlens, b, gate, nthreads, _lib_path):
    lib = _load() if _lib_path is None else _bind(_lib_path)
    arrs = [_as_array(x) for x in (q, k, v, a, beta)]
    if len({d for _, d in arrs}) != 1:
        arrs = [(np.ascontiguousarray(_widen_np(x, d)), F64) for x, d in arrs]
    (qa, dt), (ka, _), (va, _), (aa, _), (ba, _) = arrs
    B, T, H, dk = qa.shape
    dv = va.shape[-1]
    vec = fn == "gdr_oracle_bwd_vec"
    assert aa.shape == ((B, T, H, dk) if vec else (B, T, H)), aa.shape
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        assert B == 1
        N = cu.shape[0] - 1
    else:
        cu = None
        N = B

    def f64(x, shape):
        if x is None:
            return None
        xa, xd = _as_array(x)
        xa = np.ascontiguousarray(_widen_np(xa, xd))
        assert xa.shape == shape, (xa.shape, shape)
        return xa

    h0a = f64(h0, (N, H, dk, dv))
    dout_a = f64(dout, (B, T, H, dv))
    dhT_a = f64(dhT, (N, H, dk, dv))
    g = {"dq": np.zeros((B, T, H, dk)), "dk": np.zeros((B, T, H, dk)),
         "dv": np.zeros((B, T, H, dv)), "da": np.zeros((B, T, H, dk) if vec else (B, T, H)),
         "dbeta": np.zeros((B, T, H)), "dh0": np.zeros((N, H, dk, dv))}
    ptr = lambda x: None if x is None else x.ctypes.data
    rc = getattr(lib, fn)(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, aa.ctypes.data, ba.ctypes.data, dt,
        ptr(h0a), ptr(dout_a), ptr(dhT_a), g["dq"].ctypes.data, g["dk"].ctypes.data,
        g["dv"].ctypes.data, g["da"].ctypes.data, g["dbeta"].ctypes.data, g["dh0"].ctypes.data,
        None if cu is None else cu.ctypes.data, N, T, H, dk, dv, float(b), GATES[gate],
        int(nthreads))
    if rc != 0:
        raise ValueError(f"{fn} rejected its arguments (code {rc})")
    return g


def max_threads() -> int:
    return int(_load().gdr_oracle_max_threads())


def gate(a: float, b: float = 2.0, mode: str = "bounded") -> float:
    """Scalar log-decay g(a) of the oracle [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3]."""
    return float(_load().gdr_oracle_gate(float(a), float(b), GATES[mode]))


def oracle_fwd(q, k, v, a, beta, h0=None, cu_seqlens=None, b: float = 2.0,
               gate: str = "bounded", erase: bool = True, nthreads: int = 0,
               _lib_path: str | None = None):
    """Token-by-token fp64 forward.  Returns (out [B,T,H,dv], hT [N,H,dk,dv]).

    Shapes follow the library: q,k [B,T,H,dk], v [B,T,H,dv], a,beta [B,T,H];
    with cu_seqlens (N+1 offsets) B must be 1 and the N sequences are packed
    along T.  h0 is [N,H,dk,dv] (None means zero).  ``_lib_path`` loads another
    build of the C source (the mutation tests use it)."""
    return _fwd("gdr_oracle_fwd", q, k, v, a, beta, h0, cu_seqlens, b, gate, erase, nthreads,
                _lib_path)


def oracle_fwd_vec(q, k, v, a, beta, h0=None, cu_seqlens=None, b: float = 2.0,
                   gate: str = "bounded", erase: bool = True, nthreads: int = 0,
                   _lib_path: str | None = None):
    """The per-channel decay form: as ``oracle_fwd`` but a is [B,T,H,dk], one gate
    input per key channel, and row i of the state decays by exp(g(a[..., i]))."""
    return _fwd("gdr_oracle_fwd_vec", q, k, v, a, beta, h0, cu_seqlens, b, gate, erase,
                nthreads, _lib_path)


def _fwd(fn, q, k, v, a, beta, h0, cu_seqlens, b, gate, erase, nthreads, _lib_path):
    lib = _load() if _lib_path is None else _bind(_lib_path)
    arrs = [_as_array(x) for x in (q, k, v, a, beta)]
    if len({d for _, d in arrs}) != 1:
        # mixed storage: widen everything to fp64 first (exact)
        arrs = [(np.ascontiguousarray(_widen_np(x, d)), F64) for x, d in arrs]
    (qa, dt), (ka, _), (va, _), (aa, _), (ba, _) = arrs
    B, T, H, dk = qa.shape
    dv = va.shape[-1]
    want_a = (B, T, H, dk) if fn == "gdr_oracle_fwd_vec" else (B, T, H)
    assert aa.shape == want_a, (aa.shape, want_a)
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        assert B == 1
        N = cu.shape[0] - 1
    else:
        cu = None
        N = B
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((N, H, dk, dv), dtype=np.float64)
    h0a = None
    if h0 is not None:
        h0a, h0d = _as_array(h0)
        h0a = np.ascontiguousarray(_widen_np(h0a, h0d))
        assert h0a.shape == (N, H, dk, dv)
    rc = getattr(lib, fn)(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, aa.ctypes.data, ba.ctypes.data,
        dt, None if h0a is None else h0a.ctypes.data, out.ctypes.data, hT.ctypes.data,
        None if cu is None else cu.ctypes.data, N, T, H, dk, dv, float(b), GATES[gate],
        1 if erase else 0, int(nthreads))
    if rc != 0:
        raise ValueError(f"{fn} rejected its arguments (code {rc})")
    return out, hT


def _widen_np(x, code):
    if code == BF16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)
