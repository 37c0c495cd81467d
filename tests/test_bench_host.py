"""Host logic of bench.py that needs no GPU: the multi-rank timing reduction over
two gloo ranks on CPU, the per-replica workloads, the whole-job value and the
JSON line of the oracle (reference) arm."""
from __future__ import annotations

import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gdr_inputs import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, _ = bench.dist_env()
        # each rank measured a different time; everyone must see the slowest
        ms = bench.max_over_ranks(10.0 + 3.5 * rank, dist, "cpu")
        dist.barrier()
        q.put((got_rank, got_ws, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(w == ws for _, w, _ in res)
    assert all(ms == pytest.approx(13.5) for _, _, ms in res)


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(7.25, None, "cpu") == 7.25


def test_replicas_draw_distinct_inputs_of_the_same_shape():
    w = WORKLOADS["b2_t4k"]
    w0, w1 = bench.rank_workload(w, 0), bench.rank_workload(w, 1)
    assert w0 == w
    assert w1.seed != w0.seed
    assert (w1.B, w1.H, w1.T, w1.dk, w1.dv, w1.chunk, w1.dtype) == (w.B, w.H, w.T, w.dk, w.dv,
                                                                    w.chunk, w.dtype)


def test_job_value_counts_every_rank():
    # 2 ranks x 1M tokens x 4 steps in 20 ms
    assert bench.job_value(2, 1 << 20, 4, 20.0) == pytest.approx(2 * (1 << 20) * 4 / 0.02)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-tokens", "256",
                "--workload", "b2_t4k"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("b2_t4k")


# ---- the oracle timed beside the next rows' benchmark modes (CPU tensors, tiny budgets) --
def _small_inputs(T=48, B=2, H=2):
    from gdr_inputs import make_inputs
    return make_inputs(WORKLOADS["b2_t4k"].with_(B=B, H=H), device="cpu", T=T)


def _check_rate(res, cap):
    rate, n, threads, dt = res
    assert rate > 0 and dt > 0 and threads >= 1
    assert 1 <= n <= cap
    line = bench._cpu_line(rate, n, threads, dt, "sample")
    assert line["kind"] == "oracle" and line["unit"] == "tokens/s" and line["cores"] == threads
    assert str(n) in line["sample"]


def test_cpu_rate_of_the_per_channel_forward():
    from gdr_inputs import make_channel_gate
    x = _small_inputs(B=1)
    av = make_channel_gate(x, 3)
    _check_rate(bench.cpu_rate_vec(x, av, 2.0, 0.05), x["q"].shape[1])


@pytest.mark.parametrize("per_channel", [False, True])
def test_cpu_rate_of_the_backward(per_channel):
    from gdr_inputs import make_channel_gate
    x = _small_inputs()
    if per_channel:
        x["a"] = make_channel_gate(x, 4)
    dout = torch.randn(x["v"].shape).to(x["v"].dtype)
    dhT = 0.1 * torch.randn(x["h0"].shape)
    _check_rate(bench.cpu_rate_bwd(x, dout, dhT, 2.0, per_channel, 0.05), x["q"].shape[1])


def test_cpu_rate_of_the_router():
    from gdr_inputs import make_router_logits
    logits, bias = make_router_logits(512, 64, 9, "bf16", device="cpu")
    res = bench.cpu_rate_router(logits, bias, 8, 0.05)
    _check_rate(res, 512)
    assert res[2] == 1                                # the router oracle is single-threaded


def test_cpu_rate_of_one_decode_step():
    x = _small_inputs(T=1, B=4)
    _check_rate(bench.cpu_rate_decode(x, x["h0"].clone(), 2.0, 0.05), 4)
