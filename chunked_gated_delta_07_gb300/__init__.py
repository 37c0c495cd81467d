"""Chunked gated delta-rule forward pass on GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libgdr.so`` (the C ABI in ``include/gdr.h``).  It
only marshals arguments -- tensors become device pointers, streams become
``cudaStream_t`` -- and every step of the pass runs in the library's
kernels.  There is no fallback: if the library is missing, importing a
function raises.

The functions keep the C names and argument order.  ``chunk_fwd`` is a
convenience wrapper that allocates ``out`` / ``hT`` and raises on an error
status.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# GDR_LIB selects another build of the library (the checking builds of _build.py)
LIB_PATH = os.environ.get("GDR_LIB") or os.path.join(HERE, "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA = 0, 1, 2, 3
GDR_ERR_TIMEOUT, GDR_ERR_NO_WORKSPACE, GDR_ERR_BAD_SEQLENS, GDR_ERR_BOUNDS = 4, 5, 6, 7
GDR_BF16, GDR_F32 = 0, 1
GDR_GATE_BOUNDED, GDR_GATE_SOFTPLUS = 0, 1
GDR_PATH_AUTO, GDR_PATH_SIMT, GDR_PATH_TC = 0, 1, 2

EXPORTS = ("gdr_chunk_fwd", "gdr_chunk_fwd_ex", "gdr_chunk_fwd_workspace_size",
           "gdr_chunk_fwd_host", "gdr_gate_cumsum", "gdr_wy_repr", "gdr_get_status",
           "gdr_status_string", "gdr_release", "gdr_launch_count", "gdr_profile_enable",
           "gdr_profile_read", "gdr_profile_select", "gdr_chunk_fwd_noalloc", "gdr_recurrent_fwd", "gdr_chunk_bwd", "gdr_chunk_fwd_vec",
           "gdr_router_topk", "gdr_router_bias_update", "gdr_chunk_bwd_vec")

_lock = threading.Lock()
_lib = None

_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "gdr_chunk_fwd": (_I, [_P] * 9 + [_I, _I64, _I, _I, _I, _I, _F, _P]),
    "gdr_chunk_fwd_ex": (_I, [_P] * 9 + [_I, _I64, _I, _I, _I, _I, _F, _I, _I, _I, _P, _SZ, _P]),
    "gdr_chunk_fwd_workspace_size": (_SZ, [_I, _I64, _I, _I, _I, _I, _I, _I]),
    "gdr_chunk_fwd_host": (_I, [_P] * 9 + [_I, _I64, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "gdr_gate_cumsum": (_I, [_P, _P, _P, _I, _I64, _I, _I, _F, _I, _I, _P]),
    "gdr_wy_repr": (_I, [_P] * 7 + [_I, _I64, _I, _I, _I, _I, _I, _P]),
    "gdr_get_status": (_I, [_P]),
    "gdr_status_string": (ctypes.c_char_p, [_I]),
    "gdr_release": (None, []),
    "gdr_launch_count": (ctypes.c_uint64, []),
    "gdr_profile_enable": (None, [_I]),
    "gdr_profile_read": (_I, [_P, _P, _P, _I]),
    "gdr_profile_select": (None, [ctypes.c_char_p]),
    "gdr_chunk_fwd_noalloc": (_I, [_P] * 8 + [_I, _I64, _I, _I, _I, _I, _F, _I, _I, _P]),
    "gdr_recurrent_fwd": (_I, [_P] * 7 + [_I, _I64, _I, _I, _I, _F, _I, _I, _P]),
    "gdr_chunk_bwd": (_I, [_P] * 15 + [_I, _I64, _I, _I, _I, _I, _F, _I, _I, _P]),
    "gdr_chunk_fwd_vec": (_I, [_P] * 9 + [_I, _I64, _I, _I, _I, _I, _F, _I, _P]),
    "gdr_router_topk": (_I, [_P] * 5 + [_I64, _I, _I, _I, _P]),
    "gdr_router_bias_update": (_I, [_P] * 3 + [_I, _I, ctypes.c_double, ctypes.c_double, _F, _P]),
    "gdr_chunk_bwd_vec": (_I, [_P] * 15 + [_I, _I64, _I, _I, _I, _I, _F, _I, _P]),
}


class GdrError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})" if what else status_string(code))


def lib():
    """The loaded ``libgdr.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (needs nvcc)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- the C functions, same names, argument marshalling only ---------------------------
def gdr_chunk_fwd(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk, b,
                  stream=None) -> int:
    return lib().gdr_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0), _ptr(out),
                               _ptr(hT), _ptr(cu_seqlens), B, T, H, dk, dv, chunk, float(b),
                               _stream(stream))


def gdr_chunk_fwd_ex(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk, b,
                     dtype, gate, path, workspace=None, workspace_bytes=0, stream=None) -> int:
    return lib().gdr_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                                  _ptr(out), _ptr(hT), _ptr(cu_seqlens), B, T, H, dk, dv, chunk,
                                  float(b), dtype, gate, path, _ptr(workspace), workspace_bytes,
                                  _stream(stream))


def gdr_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype=GDR_BF16, path=GDR_PATH_AUTO) -> int:
    return int(lib().gdr_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype, path))


def gdr_chunk_fwd_host(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk, b,
                       dtype, gate, path, stream=None) -> int:
    """Host-buffer entry point: q..cu_seqlens are CPU tensors (pinned for full speed)."""
    return lib().gdr_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                                    _ptr(out), _ptr(hT), _ptr(cu_seqlens), B, T, H, dk, dv, chunk,
                                    float(b), dtype, gate, path, _stream(stream))


def gdr_chunk_fwd_noalloc(q, k, v, a, beta, h0, out, hT, B, T, H, dk, dv, chunk, b, dtype, gate,
                          stream=None) -> int:
    """Dense-input forward whose scratch is the library's static device array (no allocation)."""
    return lib().gdr_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                                       _ptr(out), _ptr(hT), B, T, H, dk, dv, chunk, float(b), dtype,
                                       gate, _stream(stream))


def gdr_recurrent_fwd(q, k, v, a, beta, state, out, N, T, H, dk, dv, b, dtype, gate,
                      stream=None) -> int:
    """Token-by-token form (decoding): advances state [N,H,dk,dv] in place over T tokens."""
    return lib().gdr_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(state),
                                   _ptr(out), N, T, H, dk, dv, float(b), dtype, gate, _stream(stream))


def recurrent_fwd(q, k, v, a, beta, state, b=2.0, gate="bounded", out=None, stream=None):
    """Decode T tokens: q,k [N,T,H,dk], v [N,T,H,dv], a,beta [N,T,H] on one device, state
    [N,H,dk,dv] fp32 updated in place; returns out [N,T,H,dv] (raises GdrError on failure)."""
    import torch
    if state is None:
        raise ValueError("state is required")
    N, T, H, dk, dv, _ = check_sequence_inputs(q, k, v, a, beta, h0=state, out=out)
    _require_cuda(q)
    if out is None:
        out = torch.empty((N, T, H, dv), dtype=q.dtype, device=q.device)
    rc = gdr_recurrent_fwd(q, k, v, a, beta, state, out, N, T, H, dk, dv, b, dtype_code(q),
                           _GATES[gate], stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_recurrent_fwd")
    return out


def gdr_chunk_bwd(q, k, v, a, beta, h0, dout, dhT, dq, dk, dv, da, dbeta, dh0, cu_seqlens, B, T,
                  H, dk_dim, dv_dim, chunk, b, dtype, gate, stream=None) -> int:
    """Backward pass: gradients of <dout, out> + <dhT, hT> for every input."""
    return lib().gdr_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                               _ptr(dout), _ptr(dhT), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da),
                               _ptr(dbeta), _ptr(dh0), _ptr(cu_seqlens), B, T, H, dk_dim, dv_dim,
                               chunk, float(b), dtype, gate, _stream(stream))


def gdr_chunk_fwd_vec(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk, b, dtype,
                      stream=None) -> int:
    """Forward pass with one decay factor per key channel (a is [..., H, dk])."""
    return lib().gdr_chunk_fwd_vec(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                                   _ptr(out), _ptr(hT), _ptr(cu_seqlens), B, T, H, dk, dv, chunk,
                                   float(b), dtype, _stream(stream))


def chunk_fwd_vec(q, k, v, a, beta, h0=None, cu_seqlens=None, b=2.0, want_state=True,
                  stream=None):
    """Allocate and return (out, hT) of the per-channel decay form."""
    import torch
    B, T, H, dk, dv, N = check_sequence_inputs(q, k, v, a, beta, h0, cu_seqlens, per_channel=True)
    _require_cuda(q)
    out = torch.empty_like(v)
    hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device) if want_state else None
    rc = gdr_chunk_fwd_vec(q, k, v, a, beta, h0, out, hT, cu_seqlens, N, T, H, dk, dv, 16, b,
                           dtype_code(q), stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_chunk_fwd_vec")
    return out, hT


def gdr_chunk_bwd_vec(q, k, v, a, beta, h0, dout, dhT, dq, dk, dv, da, dbeta, dh0, cu_seqlens, B,
                      T, H, dk_dim, dv_dim, chunk, b, dtype, stream=None) -> int:
    """Backward of the per-channel decay form (a and da are [..., H, dk])."""
    return lib().gdr_chunk_bwd_vec(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
                                   _ptr(dout), _ptr(dhT), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da),
                                   _ptr(dbeta), _ptr(dh0), _ptr(cu_seqlens), B, T, H, dk_dim, dv_dim,
                                   chunk, float(b), dtype, _stream(stream))


def chunk_bwd_vec(q, k, v, a, beta, dout=None, dhT=None, h0=None, cu_seqlens=None, b=2.0,
                  want_dh0=True, stream=None):
    """Allocate and return (dq, dk, dv, da, dbeta, dh0) of the per-channel form."""
    import torch
    B, T, H, dk, dv, N = check_sequence_inputs(q, k, v, a, beta, h0, cu_seqlens, per_channel=True,
                                               dout=dout, dhT=dhT)
    _require_cuda(q)
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    da, dbeta = torch.empty_like(a), torch.empty_like(beta)
    dh0 = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device) if want_dh0 else None
    rc = gdr_chunk_bwd_vec(q, k, v, a, beta, h0, dout, dhT, dq, dkk, dvv, da, dbeta, dh0,
                           cu_seqlens, N, T, H, dk, dv, 16, b, dtype_code(q), stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_chunk_bwd_vec")
    return dq, dkk, dvv, da, dbeta, dh0


GDR_QB_SIGN, GDR_QB_PROPORTIONAL = 0, 1
_QB = {"sign": GDR_QB_SIGN, "proportional": GDR_QB_PROPORTIONAL}


def gdr_router_topk(logits, bias, topk_idx, topk_logit, load, T, E, k, dtype, stream=None) -> int:
    """Top-k experts of logits + bias per token; load counts are added."""
    return lib().gdr_router_topk(_ptr(logits), _ptr(bias), _ptr(topk_idx), _ptr(topk_logit),
                                 _ptr(load), T, E, k, dtype, _stream(stream))


def gdr_router_bias_update(load, bias, thresholds, E, mode, q_lo, q_hi, eta, stream=None) -> int:
    """Quantile-balancing bias step (sign or proportional), in place on bias."""
    return lib().gdr_router_bias_update(_ptr(load), _ptr(bias), _ptr(thresholds), E, mode,
                                        float(q_lo), float(q_hi), float(eta), _stream(stream))


def router_topk(logits, bias, k, load=None, want_logits=True, stream=None):
    """Return (idx [T, k] int32, picked logits [T, k] fp32 or None); counts go to load."""
    import torch
    if logits is None or logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"logits: dtype {logits.dtype}, expected bfloat16 or float32")
    T, E = logits.shape
    _expect("logits", logits, (T, E), logits.dtype, logits.device)
    _expect("bias", bias, (E,), torch.float32, logits.device)
    if load is not None:
        _expect("load", load, (E,), torch.int64, logits.device)
    _require_cuda(logits, "logits")
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    sel = torch.empty((T, k), dtype=torch.float32, device=logits.device) if want_logits else None
    rc = gdr_router_topk(logits, bias, idx, sel, load, T, E, k, dtype_code(logits), stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_router_topk")
    return idx, sel


def router_bias_update(load, bias, mode="sign", q_lo=0.1, q_hi=0.9, eta=1e-3, stream=None):
    """Update bias in place; returns the fp64 thresholds (Q(q_lo), Q(q_hi)) on the device."""
    import torch
    if bias is None or bias.dim() != 1:
        raise ValueError("bias must be [E]")
    _expect("bias", bias, bias.shape, torch.float32, bias.device)
    _expect("load", load, bias.shape, torch.int64, bias.device)
    _require_cuda(bias, "bias")
    if mode not in _QB:
        raise ValueError(f"mode must be one of {sorted(_QB)}")
    thr = torch.empty(2, dtype=torch.float64, device=bias.device)
    rc = gdr_router_bias_update(load, bias, thr, bias.numel(), _QB[mode], q_lo, q_hi, eta, stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_router_bias_update")
    return thr


def chunk_bwd(q, k, v, a, beta, dout=None, dhT=None, h0=None, cu_seqlens=None, chunk=16, b=2.0,
              gate="bounded", want_dh0=True, stream=None):
    """Allocate and return (dq, dk, dv, da, dbeta, dh0) for tensors laid out as in chunk_fwd."""
    import torch
    B, T, H, dk, dv, N = check_sequence_inputs(q, k, v, a, beta, h0, cu_seqlens, dout=dout, dhT=dhT)
    _require_cuda(q)
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    da, dbeta = torch.empty_like(a), torch.empty_like(beta)
    dh0 = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device) if want_dh0 else None
    rc = gdr_chunk_bwd(q, k, v, a, beta, h0, dout, dhT, dq, dkk, dvv, da, dbeta, dh0, cu_seqlens,
                       N if cu_seqlens is not None else B, T, H, dk, dv, chunk, b, dtype_code(q),
                       _GATES[gate], stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_chunk_bwd")
    return dq, dkk, dvv, da, dbeta, dh0


def gdr_gate_cumsum(a, G, cu_seqlens, B, T, H, chunk, b, dtype, gate, stream=None) -> int:
    return lib().gdr_gate_cumsum(_ptr(a), _ptr(G), _ptr(cu_seqlens), B, T, H, chunk, float(b),
                                 dtype, gate, _stream(stream))


def gdr_wy_repr(k, v, beta, G, W, U, cu_seqlens, B, T, H, dk, dv, chunk, dtype, stream=None) -> int:
    return lib().gdr_wy_repr(_ptr(k), _ptr(v), _ptr(beta), _ptr(G), _ptr(W), _ptr(U),
                             _ptr(cu_seqlens), B, T, H, dk, dv, chunk, dtype, _stream(stream))


def gdr_get_status(stream=None) -> int:
    return int(lib().gdr_get_status(_stream(stream)))


def gdr_status_string(code: int) -> str:
    return lib().gdr_status_string(int(code)).decode()


def gdr_release() -> None:
    lib().gdr_release()


def gdr_launch_count() -> int:
    return int(lib().gdr_launch_count())


def gdr_profile_enable(on: bool) -> None:
    lib().gdr_profile_enable(1 if on else 0)


def gdr_profile_select(name) -> None:
    """Time only the launches of kernel `name` (None: every kernel)."""
    lib().gdr_profile_select(None if name is None else name.encode())


def gdr_profile_read(max_kernels: int = 32) -> dict:
    """{kernel name: (total ms, launches)} since the last read (clears the record)."""
    names = (ctypes.c_char_p * max_kernels)()
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int * max_kernels)()
    n = lib().gdr_profile_read(ctypes.cast(names, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                               ctypes.cast(cnt, ctypes.c_void_p), max_kernels)
    return {names[i].decode(): (float(ms[i]), int(cnt[i])) for i in range(min(n, max_kernels))}


def status_string(code: int) -> str:
    try:
        return gdr_status_string(code)
    except ImportError:
        return f"status {code}"


# ---- convenience -----------------------------------------------------------------------
_GATES = {"bounded": GDR_GATE_BOUNDED, "softplus": GDR_GATE_SOFTPLUS}
_PATHS = {"auto": GDR_PATH_AUTO, "simt": GDR_PATH_SIMT, "tc": GDR_PATH_TC}


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return GDR_BF16
    if t.dtype == torch.float32:
        return GDR_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ---- argument checks of the tensor-level calls ------------------------------------------
# The C entry points take pointers and sizes only.  The calls below take the sizes from q
# (or logits) and check every other tensor against them before the C call, so that a
# mismatched tensor raises ValueError here instead of being read out of bounds on the
# device.  Nothing here computes any part of the method.

def _expect(name, t, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device} (the device of the first input)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _require_cuda(t, name="q"):
    if not t.is_cuda:
        raise ValueError(f"{name} is on {t.device}: the library runs on CUDA devices only")


def check_sequence_inputs(q, k, v, a, beta, h0=None, cu_seqlens=None, per_channel=False,
                          dout=None, dhT=None, out=None, hT=None):
    """Check the tensors of a forward or backward call against q [B, T, H, dk]:
    k [B,T,H,dk], v [B,T,H,dv], a [B,T,H] (or [B,T,H,dk] per channel), beta [B,T,H],
    all of q's dtype (bf16 or fp32) and device, contiguous; cu_seqlens int32 [N+1] with
    B = 1; h0, hT, dhT fp32 [N,H,dk,dv]; out, dout like v.  Returns (B, T, H, dk, dv, N).
    Raises ValueError on the first mismatch (the device kind is checked by the callers)."""
    import torch
    if q is None or q.dim() != 4:
        raise ValueError("q must be [B, T, H, dk]")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"q: dtype {q.dtype}, expected bfloat16 or float32")
    B, T, H, dk = q.shape
    dev, dt = q.device, q.dtype
    _expect("q", q, (B, T, H, dk), dt, dev)
    _expect("k", k, (B, T, H, dk), dt, dev)
    if v is None or v.dim() != 4:
        raise ValueError("v must be [B, T, H, dv]")
    dv = v.shape[-1]
    _expect("v", v, (B, T, H, dv), dt, dev)
    _expect("a", a, (B, T, H, dk) if per_channel else (B, T, H), dt, dev)
    _expect("beta", beta, (B, T, H), dt, dev)
    if cu_seqlens is None:
        N = B
    else:
        if B != 1:
            raise ValueError("with cu_seqlens the token tensors are [1, T_total, H, *]")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be [N + 1] with N >= 1")
        _expect("cu_seqlens", cu_seqlens, cu_seqlens.shape, torch.int32, dev)
        N = cu_seqlens.numel() - 1
    for name, t in (("h0", h0), ("hT", hT), ("dhT", dhT)):
        if t is not None:
            _expect(name, t, (N, H, dk, dv), torch.float32, dev)
    for name, t in (("out", out), ("dout", dout)):
        if t is not None:
            _expect(name, t, (B, T, H, dv), dt, dev)
    return B, T, H, dk, dv, N


def chunk_fwd(q, k, v, a, beta, h0=None, cu_seqlens=None, chunk=16, b=2.0, gate="bounded",
              path="auto", out=None, hT=None, want_state=True, stream=None, workspace=None):
    """Allocate out (and hT), run gdr_chunk_fwd_ex, raise GdrError on a failing status.

    q,k [B,T,H,dk], v [B,T,H,dv], a,beta [B,T,H] on one CUDA device, all of one
    dtype (bf16 or fp32); with cu_seqlens (int32, N+1) B must be 1."""
    import torch
    B, T, H, dk, dv, N = check_sequence_inputs(q, k, v, a, beta, h0, cu_seqlens, out=out, hT=hT)
    _require_cuda(q)
    if workspace is not None:
        _require_cuda(workspace, "workspace")
        if workspace.device != q.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on q's device")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_state:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = gdr_chunk_fwd_ex(q, k, v, a, beta, h0, out, hT, cu_seqlens, N if cu_seqlens is not None else B,
                          T, H, dk, dv, chunk, b, dtype_code(q), _GATES[gate], _PATHS[path],
                          workspace, ws_bytes, stream)
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_chunk_fwd_ex")
    return out, hT
