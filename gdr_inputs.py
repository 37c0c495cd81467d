"""Seeded synthetic inputs for the chunked gated delta-rule forward pass.

This module is shared by the CUDA side (binding tests, bench) and the oracle
side (pins, parity).  It holds only random-number generation and input
shaping; none of the method's arithmetic (no gate, no cumsum, no recurrence)
lives here.

Workloads (the pages name no dataset; these stand in for the long-context
workloads of the 8K -> 1M context curriculum the pages describe):

  small_fp32   B=1  H=2  T=256      d=64   chunk=16  fp32   b=2  h0=0
  b2_t4k       B=2  H=16 T=4096     d=128  chunk=16  bf16   b=2  h0~N(0,0.02)
  h32_t64k     B=1  H=32 T=65536    d=128  chunk in {16,32,64}, b in {2,8},
                                                   a~N(0,2), bf16, h0=0
  t1m          B=1  H=16 T=1048576  d=128  chunk=16  bf16   b=2  h0=0
  varlen_1m    sum(T)=1048576, lengths log-uniform in [1024, 262144] (the
               last one clipped), H=16, d=128, chunk=16, bf16, h0~N(0,0.02)
               per sequence; bounded gate (b=2, a~N(0,1)) or the unbounded
               softplus gate (a~N(0,3))

Distributions (all workloads unless stated): q, k ~ N(0,1) then L2-normalised
per (token, head) in fp32 before the cast; v ~ N(0,1); beta = sigmoid(N(0,1));
gate logits a ~ N(0, std).  N(0, s) means standard deviation s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int                 # tokens per sequence (dense) or total tokens (varlen)
    dk: int = 128
    dv: int = 128
    chunk: int = 16
    dtype: str = "bf16"    # storage / arithmetic type of q, k, v, a, beta, out
    b: float = 2.0         # bound of the scaled-sigmoid gate
    gate: str = "bounded"  # or "softplus"
    a_std: float = 1.0
    a_mean: float = 0.0    # shifts the gate logits (a very negative mean = weak decay)
    h0_std: float = 0.0
    varlen: bool = False
    len_min: int = 1024
    len_max: int = 262144
    seed: int = 1000
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "small_fp32": Workload("small_fp32", B=1, H=2, T=256, dk=64, dv=64, chunk=16,
                           dtype="f32", seed=1000),
    "b2_t4k": Workload("b2_t4k", B=2, H=16, T=4096, h0_std=0.02, seed=1001),
    "h32_t64k": Workload("h32_t64k", B=1, H=32, T=65536, a_std=2.0, seed=1002),
    "t1m": Workload("t1m", B=1, H=16, T=1 << 20, seed=1003),
    "varlen_1m": Workload("varlen_1m", B=1, H=16, T=1 << 20, h0_std=0.02,
                          varlen=True, seed=1004),
}


def h32_variant(chunk: int, b: float) -> Workload:
    """The chunk / gate-bound sweep of the 32-head 64K-token workload."""
    idx = {16: 0, 32: 1, 64: 2}[chunk]
    w = WORKLOADS["h32_t64k"]
    return w.with_(name=f"h32_t64k_c{chunk}_b{int(b)}", chunk=chunk, b=float(b),
                   seed=w.seed + 10 * idx + int(b))


def softplus_variant(w: Workload) -> Workload:
    """The same shapes with the unbounded gate and a ~ N(0, 3)."""
    return w.with_(name=w.name + "_softplus", gate="softplus", a_std=3.0)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Sequence lengths drawn log-uniformly in [lo, hi] until they cover total;
    the last one is clipped so that the lengths sum to exactly total."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    lens: list[int] = []
    acc = 0
    while acc < total:
        u = torch.rand((), generator=g, dtype=torch.float64).item()
        n = int(round(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def make_inputs(w: Workload, device="cpu", T: int | None = None, block: int = 1 << 16):
    """Draw the workload's tensors on ``device`` (seeded, deterministic per device).

    Returns a dict with q, k, v, a, beta (storage dtype), h0 (fp32 or None),
    cu_seqlens (int32 or None) and the shape parameters.  ``T`` overrides the
    per-sequence (or total) token count, for reduced-size parity cases.
    """
    device = torch.device(device)
    T = w.T if T is None else T
    dt = torch_dtype(w.dtype)
    g = torch.Generator(device=device).manual_seed(w.seed)
    if w.varlen:
        lens = varlen_lengths(T, min(w.len_min, T), min(w.len_max, T), w.seed)
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        B, Tt, N = 1, T, len(lens)
    else:
        cu = None
        B, Tt, N = w.B, T, w.B
    H, dk, dv = w.H, w.dk, w.dv
    q = torch.empty((B, Tt, H, dk), dtype=dt, device=device)
    k = torch.empty((B, Tt, H, dk), dtype=dt, device=device)
    v = torch.empty((B, Tt, H, dv), dtype=dt, device=device)
    a = torch.empty((B, Tt, H), dtype=dt, device=device)
    beta = torch.empty((B, Tt, H), dtype=dt, device=device)
    # draw in token blocks so that full-size workloads never hold fp32 copies
    for bi in range(B):
        for t0 in range(0, Tt, block):
            t1 = min(Tt, t0 + block)
            n = t1 - t0
            x = _randn((n, H, dk), g, device)
            q[bi, t0:t1] = (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(dt)
            x = _randn((n, H, dk), g, device)
            k[bi, t0:t1] = (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(dt)
            v[bi, t0:t1] = _randn((n, H, dv), g, device).to(dt)
            beta[bi, t0:t1] = torch.sigmoid(_randn((n, H), g, device)).to(dt)
            a[bi, t0:t1] = (w.a_mean + w.a_std * _randn((n, H), g, device)).to(dt)
    h0 = None
    if w.h0_std > 0:
        h0 = (w.h0_std * _randn((N, H, dk, dv), g, device)).contiguous()
    if cu is not None:
        cu = cu.to(device)
    return dict(q=q, k=k, v=v, a=a, beta=beta, h0=h0, cu_seqlens=cu, B=B, T=Tt,
                N=N, H=H, dk=dk, dv=dv, chunk=w.chunk, b=w.b, gate=w.gate, dtype=w.dtype)


def make_channel_gate(x: dict, seed: int, a_std: float = 1.0, a_mean: float = 0.0,
                      block: int = 1 << 14):
    """Gate inputs of the per-channel decay form: a [B, T, H, dk] in x's storage
    dtype on x's device, ~ N(a_mean, a_std^2), drawn in token blocks."""
    q = x["q"]
    B, T, H, dk = q.shape
    g = torch.Generator(device=q.device).manual_seed(seed)
    a = torch.empty((B, T, H, dk), dtype=q.dtype, device=q.device)
    for bi in range(B):
        for t0 in range(0, T, block):
            t1 = min(T, t0 + block)
            a[bi, t0:t1] = (a_mean + a_std * _randn((t1 - t0, H, dk), g, q.device)).to(q.dtype)
    return a


def make_router_logits(T: int, E: int, seed: int, dtype: str = "bf16", device="cpu",
                       skew: float = 1.0, ties: bool = False, block: int = 1 << 16):
    """Synthetic routing logits [T, E]: N(0, 1) plus a fixed per-expert offset of
    scale ``skew`` (drawn once), so that some experts are systematically
    over-picked -- the imbalance the bias update corrects.  ``ties`` rounds the
    logits to multiples of 1/2 (many equal scores).  Also returns a bias [E] fp32
    ~ N(0, 0.01^2)."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed)
    dt = torch_dtype(dtype)
    off = skew * _randn((E,), g, device)
    x = torch.empty((T, E), dtype=dt, device=device)
    for t0 in range(0, T, block):
        t1 = min(T, t0 + block)
        y = _randn((t1 - t0, E), g, device) + off
        if ties:
            y = torch.round(y * 2) / 2
        x[t0:t1] = y.to(dt)
    bias = 0.01 * _randn((E,), g, device)
    return x, bias
