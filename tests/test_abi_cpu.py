"""The C ABI library loads, exports every declared symbol and rejects bad
arguments before touching the GPU (CPU only: no compute call runs here)."""
import os
import re

import pytest

import chunked_gated_delta_07_gb300 as gdr
from chunked_gated_delta_07_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    _build.build()
    return gdr.lib()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^GDR_API\s+[^;(]*?\b(gdr_\w+)\s*\(", text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gdr.EXPORTS)


def test_status_strings(lib):
    for code in range(8):
        assert gdr.gdr_status_string(code)
    assert gdr.gdr_status_string(99) == "unknown status"


def _call(**kw):
    base = dict(q=1 << 20, k=2 << 20, v=3 << 20, a=4 << 20, beta=5 << 20, h0=None, out=6 << 20,
                hT=None, cu_seqlens=None, B=1, T=64, H=2, dk=128, dv=128, chunk=16, b=2.0,
                dtype=gdr.GDR_BF16, gate=gdr.GDR_GATE_BOUNDED, path=gdr.GDR_PATH_AUTO,
                workspace=None, workspace_bytes=0, stream=0)
    base.update(kw)
    return gdr.gdr_chunk_fwd_ex(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), gdr.GDR_ERR_INVALID_ARG),
    (dict(H=0), gdr.GDR_ERR_INVALID_ARG),
    (dict(T=-1), gdr.GDR_ERR_INVALID_ARG),
    (dict(dk=96), gdr.GDR_ERR_UNSUPPORTED),
    (dict(dv=256), gdr.GDR_ERR_UNSUPPORTED),
    (dict(chunk=8), gdr.GDR_ERR_UNSUPPORTED),
    (dict(chunk=0), gdr.GDR_ERR_INVALID_ARG),
    (dict(b=0.0), gdr.GDR_ERR_INVALID_ARG),
    (dict(b=float("inf")), gdr.GDR_ERR_INVALID_ARG),
    (dict(b=float("nan")), gdr.GDR_ERR_INVALID_ARG),
    (dict(dtype=7), gdr.GDR_ERR_INVALID_ARG),
    (dict(gate=3), gdr.GDR_ERR_INVALID_ARG),
    (dict(path=9), gdr.GDR_ERR_INVALID_ARG),
    (dict(q=None), gdr.GDR_ERR_INVALID_ARG),
    (dict(out=None), gdr.GDR_ERR_INVALID_ARG),
    (dict(out=1 << 20), gdr.GDR_ERR_INVALID_ARG),          # out aliases q
    (dict(hT=(5 << 20) + 8), gdr.GDR_ERR_INVALID_ARG),     # hT overlaps beta
    (dict(h0=7 << 20, hT=(7 << 20) + 4), gdr.GDR_ERR_INVALID_ARG),  # partial h0/hT overlap
    (dict(q=1 << 52, k=2 << 52, v=3 << 52, a=4 << 52, beta=5 << 52, out=6 << 52, T=1 << 40,
          H=1 << 22), gdr.GDR_ERR_UNSUPPORTED),                 # > 2^40 (token, head) rows
])
def test_bad_arguments_are_rejected_before_launch(lib, kw, code):
    assert _call(**kw) == code


def test_softplus_ignores_b(lib):
    # b is not checked for the unbounded gate; the call still fails only on the
    # missing q (proves the b check was skipped)
    assert _call(gate=gdr.GDR_GATE_SOFTPLUS, b=0.0, q=None) == gdr.GDR_ERR_INVALID_ARG


def test_workspace_size(lib):
    n = gdr.gdr_chunk_fwd_workspace_size(2, 4096, 16, 128, 128, 16, gdr.GDR_BF16, gdr.GDR_PATH_SIMT)
    # at least G plus W and U in fp32
    assert n >= 4 * 2 * 4096 * 16 * (1 + 128 + 128)
    assert gdr.gdr_chunk_fwd_workspace_size(0, 4096, 16, 128, 128, 16, gdr.GDR_BF16, 0) == 0
    assert gdr.gdr_chunk_fwd_workspace_size(1, 4096, 16, 96, 128, 16, gdr.GDR_BF16, 0) == 0


def test_launch_count_starts_at_zero_without_calls(lib):
    assert gdr.gdr_launch_count() >= 0


def test_tc_path_needs_aligned_q_k_v(lib):
    # the tensor-core path reads q, k, v as TMA tiles: an explicit request with an
    # unaligned one is unsupported (AUTO runs the CUDA-core kernels instead)
    for name in ("q", "k", "v"):
        bad = {name: dict(q=1 << 20, k=2 << 20, v=3 << 20)[name] + 2}
        assert _call(path=gdr.GDR_PATH_TC, **bad) == gdr.GDR_ERR_UNSUPPORTED, name


def test_workspace_size_auto_covers_both_paths(lib):
    args = (2, 4096, 16, 128, 128, 16, gdr.GDR_BF16)
    auto = gdr.gdr_chunk_fwd_workspace_size(*args, gdr.GDR_PATH_AUTO)
    assert auto >= gdr.gdr_chunk_fwd_workspace_size(*args, gdr.GDR_PATH_TC) > 0
    assert auto >= gdr.gdr_chunk_fwd_workspace_size(*args, gdr.GDR_PATH_SIMT) > 0


def test_recurrent_state_must_be_aligned(lib):
    base = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20]
    args = (1, 1, 2, 128, 128, 2.0, gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED, 0)
    assert gdr.gdr_recurrent_fwd(*base, (7 << 20) + 4, 6 << 20, *args) == gdr.GDR_ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["dhT", "dh0"])
def test_backward_state_gradients_must_be_aligned(lib, which):
    # T = 0: the call would only copy dhT to dh0, but the check comes first
    ptr = {"dhT": 8 << 20, "dh0": 9 << 20}
    ptr[which] += 8
    ins = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, None, 6 << 20, ptr["dhT"]]
    outs = [10 << 20, 11 << 20, 12 << 20, 13 << 20, 14 << 20, ptr["dh0"]]
    rc = gdr.gdr_chunk_bwd(*ins, *outs, None, 1, 0, 2, 128, 128, 16, 2.0, gdr.GDR_BF16,
                           gdr.GDR_GATE_BOUNDED, 0)
    assert rc == gdr.GDR_ERR_INVALID_ARG


def _noalloc(**kw):
    base = dict(q=1 << 20, k=2 << 20, v=3 << 20, a=4 << 20, beta=5 << 20, h0=None, out=6 << 20,
                hT=None, B=1, T=64, H=2, dk=128, dv=128, chunk=16, b=2.0, dtype=gdr.GDR_BF16,
                gate=gdr.GDR_GATE_BOUNDED, stream=0)
    base.update(kw)
    return gdr.gdr_chunk_fwd_noalloc(*base.values())


# fake addresses 2^52 apart, so that large sizes do not make the buffers overlap
_FAR = dict(q=1 << 52, k=2 << 52, v=3 << 52, a=4 << 52, beta=5 << 52, out=6 << 52)


@pytest.mark.parametrize("kw,code", [
    # sizes whose scratch exceeds the static array
    (dict(_FAR, T=1 << 20, H=16), gdr.GDR_ERR_NO_WORKSPACE),
    (dict(_FAR, T=1 << 20, H=1 << 20), gdr.GDR_ERR_NO_WORKSPACE),
    (dict(_FAR, B=1 << 20, T=1 << 20, H=1), gdr.GDR_ERR_NO_WORKSPACE),
    # more than 2^40 (token, head) rows, whose byte counts would wrap 64 bits
    # (2^40 tokens x 2^22 heads): refused as by the regular entry point
    (dict(_FAR, T=1 << 40, H=1 << 22), gdr.GDR_ERR_UNSUPPORTED),
    (dict(_FAR, B=1 << 20, T=1 << 20, H=1 << 30), gdr.GDR_ERR_UNSUPPORTED),
    (dict(B=1 << 30, T=0), gdr.GDR_ERR_NO_WORKSPACE),
    # the regular entry point's refusals, reached the same way
    (dict(T=(1 << 40) + 1), gdr.GDR_ERR_UNSUPPORTED),
    (dict(out=1 << 20), gdr.GDR_ERR_INVALID_ARG),                   # out aliases q
    (dict(hT=(5 << 20) + 8), gdr.GDR_ERR_INVALID_ARG),              # hT overlaps beta
    (dict(h0=7 << 20, hT=(7 << 20) + 4), gdr.GDR_ERR_INVALID_ARG),  # partial h0/hT overlap
    (dict(b=float("inf")), gdr.GDR_ERR_INVALID_ARG),
    (dict(chunk=8), gdr.GDR_ERR_UNSUPPORTED),
    (dict(q=None), gdr.GDR_ERR_INVALID_ARG),
])
def test_noalloc_refuses_before_launch(lib, kw, code):
    # fake addresses: every case is refused by the host checks, nothing is launched
    assert _noalloc(**kw) == code


def test_noalloc_refuses_what_the_regular_entry_point_refuses(lib):
    for kw in (dict(out=1 << 20), dict(hT=(5 << 20) + 8), dict(h0=7 << 20, hT=(7 << 20) + 4),
               dict(B=0), dict(dk=96), dict(b=float("nan"))):
        assert _noalloc(**kw) == _call(**kw) != gdr.GDR_OK, kw


def test_tc_path_tiles_by_16_for_every_chunk(lib):
    # bf16, d = 128: the tensor-core path takes chunk 16, 32 and 64 and runs all of them
    # on 16-token tiles (the same scratch); the CUDA-core path's scratch follows chunk
    for B, T in [(2, 4096), (3, 1000)]:
        tc = [gdr.gdr_chunk_fwd_workspace_size(B, T, 16, 128, 128, c, gdr.GDR_BF16, gdr.GDR_PATH_TC)
              for c in (16, 32, 64)]
        assert tc[0] > 0 and tc[0] == tc[1] == tc[2]
    # fp32 has no tensor-core path at any chunk
    assert gdr.gdr_chunk_fwd_workspace_size(2, 4096, 16, 128, 128, 32, gdr.GDR_F32, gdr.GDR_PATH_TC) == 0
