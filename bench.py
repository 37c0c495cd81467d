"""Benchmark of the chunked gated delta-rule forward pass (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload t1m] [--path auto|simt|tc] [--no-e2e] [--no-cpu]

A step is one full forward pass (plan, gate + cumsum, in-tile WY, state pass,
outputs) over one batch of synthetic input already resident in HBM.  The
default workload is 1,048,576 tokens x 16 heads, dk = dv = 128, tile 16, bf16,
bounded gate b = 2 (its inputs are 12.9 GB, far larger than the 129 MB L2, so
no flush is needed between steps).  Under torchrun every rank runs its own
replica on its own GPU (weak scaling, no collective on the data path); rank 0
prints the line with the max-over-ranks time.

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on
a bounded prefix of the same workload per step, and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and % roofline, gated-delta-rule chunk fwd at T=1M, H=16, d=128, bf16"
UNIT = "tokens/s"

# DRAM bytes (read + write) per launch of the dominant kernel as counted by ncu,
# per (token, head) unit, with the hash of the kernel source they were taken at.
# The value is reported only while the source is unchanged.
NCU_TRAFFIC = {
    # ncu --set full, t1m shape cut to 262,144 tokens (4,194,304 units, inputs 3.2 GB > L2):
    # dram__bytes_read.sum 3.268876 GB + dram__bytes_write.sum 1.053422 GB per launch
    "tc_output_kernel": {"source": "gdr_tc.cu", "hash": "e2d6e1dd01eb", "workload": "t1m",
                         "bytes_per_unit": 4322297600.0 / 4194304},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic(w, n_tokens, with_h0):
    """Bytes and FLOPs one pass must move / do: q, k, v, out, a, beta per
    (token, head), the final state, and h0 when given."""
    es = 2 if w.dtype == "bf16" else 4
    per_tok = es * (2 * w.dk + 2 * w.dv) + 2 * es
    nstate = (w.B if not w.varlen else 1) * w.H * w.dk * w.dv * 4
    byt = per_tok * n_tokens * w.H + nstate * (2 if with_h0 else 1)
    flops = (6 * w.chunk * w.dk + 4 * w.chunk * w.dv + 6 * w.dk * w.dv) * n_tokens * w.H
    return byt, flops, per_tok


def kernel_breakdown(gdr, torch, step, n=2):
    """Per-kernel device times over n untimed steps with every launch bracketed by
    events: ({kernel: (ms_total, launches)}, name of the largest).  The timed region
    that follows brackets the launches of that one kernel only, so that no events sit
    between the step's other launches."""
    gdr.gdr_profile_select(None)
    gdr.gdr_profile_read()
    gdr.gdr_profile_enable(True)
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    gdr.gdr_profile_enable(False)
    prof = gdr.gdr_profile_read()
    dom = max(prof.items(), key=lambda kv: kv[1][0])[0] if prof else None
    return prof, dom


def kernels_json(prof, n):
    return {k: {"ms_per_step": v[0] / n, "launches_per_step": v[1] / n} for k, v in prof.items()}


KERNELS_NOTE = ("per-kernel times from 2 untimed steps with every launch bracketed by events; "
                "the timed region brackets the dominant kernel's launches only")


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except (ValueError, IndexError):
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w, rank):
    """Each replica draws its own inputs: same shapes, seed offset by rank."""
    return w.with_(seed=w.seed + 7919 * rank)


def max_over_ranks(ms, dist, device):
    """The timed region's length as the slowest rank measured it."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ws, n_tokens, steps, ms):
    """Whole-job tokens/s: every rank processed n_tokens per step."""
    return ws * n_tokens * steps / (ms / 1e3)


def cpu_oracle_rate(x, w, budget_s, max_tokens):
    """Time the oracle on a prefix of the workload; returns (tokens/s, tokens, threads, seconds)."""
    import oracle
    threads = oracle.max_threads()

    def run(n):
        sl = {k: x[k][:, :n].cpu() for k in ("q", "k", "v", "a", "beta")}
        t0 = time.perf_counter()
        oracle.oracle_fwd(sl["q"], sl["k"], sl["v"], sl["a"], sl["beta"], h0=None, b=w.b,
                          gate=w.gate, nthreads=threads)
        return time.perf_counter() - t0

    nseq = x["q"].shape[0]   # dense input: the prefix of every sequence
    n = 256
    dt = run(n)
    n = int(min(max_tokens // nseq, x["q"].shape[1], max(256, n * budget_s / max(dt, 1e-6) / nseq)))
    dt = run(n)
    return nseq * n / dt, nseq * n, threads, dt


def _grow_to_budget(run, n_min, budget_s, n_max):
    """Time run(n) on n_min units, then on as many as fit the budget (at most n_max);
    returns (units/s, units, seconds)."""
    n = n_min
    dt = run(n)
    n = int(min(n_max, max(n_min, n * budget_s / max(dt, 1e-6))))
    dt = run(n)
    return n / dt, n, dt


def cpu_rate_vec(x, av, b, budget_s):
    """The per-channel oracle on the first n tokens of every head (packed tokens taken
    as one sequence); returns (tokens/s, tokens, threads, seconds)."""
    import oracle
    threads = oracle.max_threads()

    def run(n):
        sl = [t[:, :n].cpu() for t in (x["q"], x["k"], x["v"], av, x["beta"])]
        t0 = time.perf_counter()
        oracle.oracle_fwd_vec(*sl, h0=None, b=b, nthreads=threads)
        return time.perf_counter() - t0

    rate, n, dt = _grow_to_budget(run, 64, budget_s, x["q"].shape[1])
    return rate, n, threads, dt


def cpu_rate_bwd(x, dout, dhT, b, per_channel, budget_s):
    """The oracle backward on the first n tokens of sequence 0, every head (the
    per-channel oracle keeps every state, so n <= 1024 there); returns
    (tokens/s, tokens, threads, seconds)."""
    import oracle
    threads = oracle.max_threads()
    fn = oracle.oracle_bwd_vec if per_channel else oracle.oracle_bwd

    def run(n):
        sl = [t[:1, :n].cpu() for t in (x["q"], x["k"], x["v"], x["a"], x["beta"], dout)]
        h0 = None if x["h0"] is None else x["h0"][:1].cpu()
        d_t = dhT[:1].cpu()
        t0 = time.perf_counter()
        fn(*sl[:5], dout=sl[5], dhT=d_t, h0=h0, b=b, nthreads=threads)
        return time.perf_counter() - t0

    cap = min(x["q"].shape[1], 1024 if per_channel else x["q"].shape[1])
    rate, n, dt = _grow_to_budget(run, 32, budget_s, cap)
    return rate, n, threads, dt


def cpu_rate_router(logits, bias, k, budget_s):
    """The router oracle (top-k of logit + bias, counts) on the first n tokens of the
    window; returns (tokens/s, tokens, threads, seconds)."""
    import oracle

    def run(n):
        sl = logits[:n].cpu()
        bz = bias.cpu()
        t0 = time.perf_counter()
        oracle.router_topk(sl, bz, k)
        return time.perf_counter() - t0

    rate, n, dt = _grow_to_budget(run, 256, budget_s, logits.shape[0])
    return rate, n, 1, dt


def cpu_rate_decode(x, state, b, budget_s):
    """The oracle on one decode step of the first n sequences, every head; returns
    (tokens/s, tokens, threads, seconds)."""
    import oracle
    threads = oracle.max_threads()

    def run(n):
        sl = [t[:n].cpu() for t in (x["q"], x["k"], x["v"], x["a"], x["beta"])]
        h = state[:n].cpu()
        t0 = time.perf_counter()
        oracle.oracle_fwd(*sl, h0=h, b=b, nthreads=threads)
        return time.perf_counter() - t0

    rate, n, dt = _grow_to_budget(run, 1, budget_s, x["q"].shape[0])
    return rate, n, threads, dt


def _cpu_line(rate, n, threads, dt, what):
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{what}: {n} tokens, fp64 oracle, {dt:.1f} s"}


def bench_reference(args, w):
    """The oracle arm: fp64 CPU oracle, a bounded prefix of the workload per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import torch

    from gdr_inputs import make_inputs
    threads = oracle.max_threads()
    per_step_tokens = max(256, args.ref_tokens)
    x = make_inputs(w, device="cpu", T=per_step_tokens)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.oracle_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], h0=x["h0"], b=w.b, gate=w.gate,
                          nthreads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = per_step_tokens * args.steps / tot
    sample = (f"first {per_step_tokens} tokens of each of the {w.H} heads of workload {w.name} per step "
              f"(fp64, token by token)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w):
    shape = (f"varlen total={w.T}" if w.varlen else f"B={w.B} T={w.T}")
    es = 2 if w.dtype == "bf16" else 4
    in_bytes = w.T * (1 if w.varlen else w.B) * w.H * es * (2 * w.dk + w.dv + 2)
    return {"workload": f"{w.name}: {shape} H={w.H} dk={w.dk} dv={w.dv} chunk={w.chunk} "
                        f"{w.dtype} gate={w.gate} b={w.b}",
            "tokens_per_step": w.T * (1 if w.varlen else w.B), "heads": w.H,
            "l2_policy": ("inputs larger than L2 (no flush)" if in_bytes >= 2 * L2_BYTES else
                          "L2 flushed between steps (each step timed alone)")}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="t1m")
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-tokens", type=int, default=16384, help="tokens per reference step")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the tokens per sequence (or total, varlen) of the workload")
    ap.add_argument("--mode", default="prefill", choices=["prefill", "decode", "backward", "vec", "router"],
                    help="prefill: the chunked forward (the headline); decode: one recurrent "
                         "step of --decode-seqs sequences; backward: gdr_chunk_bwd on "
                         "--bwd-seqs sequences of --bwd-tokens tokens; vec: the per-channel "
                         "decay forward on --workload; router: one quantile-balancing window of "
                         "--router-tokens tokens over 896 experts")
    ap.add_argument("--router-tokens", type=int, default=1 << 20)
    ap.add_argument("--router-k", type=int, default=8)
    ap.add_argument("--decode-seqs", type=int, default=256)
    ap.add_argument("--bwd-seqs", type=int, default=8)
    ap.add_argument("--bwd-tokens", type=int, default=4096)
    ap.add_argument("--bwd-per-channel", action="store_true",
                    help="backward of the per-channel decay form (gdr_chunk_bwd_vec)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    return args


def resolve_workload(name):
    """A workload by name: the five named ones, h32_t64k_c{16,32,64}_b{2,8} (the chunk and
    gate-bound sweep of the 32-head workload) and <name>_softplus (the unbounded gate)."""
    from gdr_inputs import WORKLOADS, h32_variant, softplus_variant
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.endswith("_softplus"):
        return softplus_variant(resolve_workload(name[:-len("_softplus")]))
    if name.startswith("h32_t64k_c"):
        c, b = name[len("h32_t64k_c"):].split("_b")
        return h32_variant(int(c), float(b))
    raise SystemExit(f"unknown workload {name}")


L2_BYTES = 129 * 2 ** 20


def main(argv=None):
    args = parse_args(argv)

    w = resolve_workload(args.workload)
    if args.tokens > 0:
        w = w.with_(T=args.tokens)
    if args.impl == "reference":
        bench_reference(args, w)
        return
    if args.mode == "decode":
        bench_decode(args)
        return
    if args.mode == "backward":
        bench_backward(args)
        return
    if args.mode == "vec":
        bench_vec(args, w)
        return
    if args.mode == "router":
        bench_router(args)
        return

    import torch
    import chunked_gated_delta_07_gb300 as gdr
    from gdr_inputs import make_inputs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    gdr.lib()

    x = make_inputs(rank_workload(w, rank), device=dev)
    B, T, H, dk, dv = x["B"], x["T"], x["H"], x["dk"], x["dv"]
    N = x["N"]
    n_tokens = T if w.varlen else B * T
    out = torch.empty_like(x["v"])
    hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    dcode = gdr.GDR_BF16 if w.dtype == "bf16" else gdr.GDR_F32
    gcode = gdr.GDR_GATE_BOUNDED if w.gate == "bounded" else gdr.GDR_GATE_SOFTPLUS
    pcode = {"auto": gdr.GDR_PATH_AUTO, "simt": gdr.GDR_PATH_SIMT, "tc": gdr.GDR_PATH_TC}[args.path]
    stream = torch.cuda.current_stream(dev)

    def step():
        rc = gdr.gdr_chunk_fwd_ex(x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], out, hT,
                                  x["cu_seqlens"], N, T, H, dk, dv, w.chunk, w.b, dcode, gcode,
                                  pcode, None, 0, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_chunk_fwd_ex")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = gdr.gdr_get_status(stream)
    if st != gdr.GDR_OK:
        raise gdr.GdrError(st, "device status after warm-up")

    # ---- timed region ----
    # Inputs smaller than twice the L2 are timed step by step, with the L2 flushed
    # (a buffer of twice its size written) between steps, outside the timed steps.
    in_bytes = sum(t.numel() * t.element_size() for t in (x["q"], x["k"], x["v"], x["a"], x["beta"]))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if in_bytes < 2 * L2_BYTES else None
    breakdown, dom_sel = kernel_breakdown(gdr, torch, step)
    gdr.gdr_profile_select(dom_sel)
    gdr.gdr_profile_read()           # drop anything recorded so far
    gdr.gdr_profile_enable(True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush is not None else 1)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        n_launch0 = gdr.gdr_launch_count()
        if flush is None:
            evs[0][0].record(stream)
            for _ in range(args.steps):
                step()
            evs[0][1].record(stream)
        else:
            for e0, e1 in evs:
                flush.fill_(1.0)
                e0.record(stream)
                step()
                e1.record(stream)
        torch.cuda.synchronize()
        n_launch = gdr.gdr_launch_count() - n_launch0
    gdr.gdr_profile_enable(False)
    gdr.gdr_profile_select(None)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    ms = max_over_ranks(ms, dist, dev)
    if dist:
        dist.barrier()
    prof = gdr.gdr_profile_read()
    st = gdr.gdr_get_status(stream)
    if st != gdr.GDR_OK:
        raise gdr.GdrError(st, "device status after timed region")

    ms_step = ms / args.steps
    value = job_value(ws, n_tokens, args.steps, ms)
    hbm, tf_burst, tf_sust, peak_src = peaks()
    byt, flops, per_tok = algorithmic(w, n_tokens, x["h0"] is not None)
    t_roof = max(byt / (hbm * 1e9), flops / (tf_sust * 1e12))
    step_frac = t_roof / (ms_step / 1e3)

    # dominant kernel: largest summed device time in the timed region
    dom_name, (dom_ms, dom_n) = max(prof.items(), key=lambda kv: kv[1][0]) if prof else ("?", (0.0, 1))
    dom_avg_s = dom_ms / max(dom_n, 1) / 1e3
    units = n_tokens * H                                  # (token, head) units per launch
    achieved = per_tok * units / dom_avg_s / 1e9 if dom_avg_s > 0 else 0.0
    traffic = None
    rec = NCU_TRAFFIC.get(dom_name)
    if rec:
        src = os.path.join(ROOT, "chunked_gated_delta_07_gb300", "csrc", rec["source"])
        if os.path.exists(src) and source_hash(src) == rec["hash"] and rec.get("workload") == w.name:
            traffic = rec["bytes_per_unit"] * units
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "kernel": dom_name,
                "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_unit": per_tok, "units_per_launch": units,
                "kernel_avg_ms": dom_avg_s * 1e3,
                "kernel_share": (breakdown[dom_name][0] / sum(v[0] for v in breakdown.values())
                                 if dom_name in breakdown else None)}

    # ---- end to end through the host-buffer entry point ----
    e2e = None
    if not args.no_e2e and rank == 0:
        e2e = bench_e2e(gdr, torch, x, w, args, dcode, gcode, pcode, n_tokens)

    cpu = None
    if not args.no_cpu and rank == 0 and ws == 1:
        rate, ntok, threads, secs = cpu_oracle_rate(x, w, args.cpu_budget, n_tokens)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {ntok // x['q'].shape[0]} tokens of each of {x['q'].shape[0]} sequence(s) x {H} heads of workload {w.name}, fp64 oracle, "
                         f"{secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w), parallelism=f"replicas x{ws}", path=args.path),
            "pct_roofline": 100.0 * step_frac,
            "step_roofline": {"t_roof_ms": t_roof * 1e3, "bytes": byt, "flops": flops,
                              "hbm_gbs": hbm, "bf16_tflops": tf_sust, "peak_source": peak_src},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_launch,
            "kernels": kernels_json(breakdown, 2), "kernels_note": KERNELS_NOTE,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def bench_decode(args):
    """One decode step (gdr_recurrent_fwd, T = 1) of N sequences x 16 heads, d = 128, bf16:
    bound by reading and writing the fp32 state (268 MB at N = 256, larger than L2)."""
    import torch
    import chunked_gated_delta_07_gb300 as gdr
    N, H, d = args.decode_seqs, 16, 128
    from gdr_inputs import WORKLOADS, make_inputs   # the t1m recipe, one token per sequence
    x = make_inputs(WORKLOADS["t1m"].with_(B=N, h0_std=0.02, seed=4000), device="cuda", T=1)
    state = x["h0"].clone()
    out = torch.empty_like(x["v"])
    stream = torch.cuda.current_stream()

    def step():
        rc = gdr.gdr_recurrent_fwd(x["q"], x["k"], x["v"], x["a"], x["beta"], state, out, N, 1, H,
                                   d, d, 2.0, gdr.GDR_BF16, gdr.GDR_GATE_BOUNDED, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_recurrent_fwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, 20)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        n0 = gdr.gdr_launch_count()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        n_launch = gdr.gdr_launch_count() - n0
    st = gdr.gdr_get_status(stream)
    if st != gdr.GDR_OK:
        raise gdr.GdrError(st, "device status after decode")
    ms = ev0.elapsed_time(ev1) / steps
    hbm, _, _, peak_src = peaks()
    byt = 2 * N * H * d * d * 4 + N * H * (4 * d * 2 + 2 * 2)   # state in + out, q k v out, a beta
    achieved = byt / (ms / 1e3) / 1e9
    cpu = None if args.no_cpu else _cpu_line(*cpu_rate_decode(x, state, 2.0, args.cpu_budget),
                                             "one decode step of the first sequences x 16 heads")
    print(json.dumps({
        "metric": "decode tokens/s, one recurrent step, 16 heads, d=128, bf16, fp32 state",
        "value": N / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode: N={N} sequences x H={H}, dk=dv={d}, T=1 per step",
                   "l2_policy": "state larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None, "kernel": "recurrent_kernel",
                     "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_step": byt},
        "cpu_baseline": cpu,
        "gpu_launches": n_launch, "clocks": clk.summary(),
    }), flush=True)


def bench_backward(args):
    """The backward pass (gdr_chunk_bwd) of N sequences x 16 heads x T tokens, d = 128,
    bf16, with h0, dout and dhT given: the chunked form on the tensor cores (tf32
    operands).  Its algorithmic work is counted as 20 dk dv flops per (token, head):
    the forward recomputed (prediction and state update) and the adjoint recurrence
    (dH, dq, ddelta, dk, dHb, dalpha and the decay of dH).  The roofline takes the
    whole step against the tf32 tensor rate (the measured bf16 rate x 1/2, the
    nominal tf32 : bf16 ratio)."""
    import torch
    import chunked_gated_delta_07_gb300 as gdr
    from gdr_inputs import WORKLOADS, make_inputs
    N, T, H, d = args.bwd_seqs, args.bwd_tokens, 16, 128
    from gdr_inputs import make_channel_gate
    x = make_inputs(WORKLOADS["t1m"].with_(B=N, h0_std=0.02, seed=4500), device="cuda", T=T)
    vec = args.bwd_per_channel
    if vec:
        x["a"] = make_channel_gate(x, 4502)
    g = torch.Generator(device="cuda").manual_seed(4501)
    dout = torch.randn(x["v"].shape, generator=g, device="cuda").to(torch.bfloat16)
    dhT = 0.1 * torch.randn((N, H, d, d), generator=g, device="cuda")
    outs = [torch.empty_like(x[n]) for n in ("q", "k", "v", "a", "beta")]
    dh0 = torch.empty_like(dhT)
    stream = torch.cuda.current_stream()

    def step():
        if vec:
            rc = gdr.gdr_chunk_bwd_vec(x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], dout,
                                       dhT, *outs, dh0, None, N, T, H, d, d, 16, 2.0, gdr.GDR_BF16,
                                       stream)
        else:
            rc = gdr.gdr_chunk_bwd(x["q"], x["k"], x["v"], x["a"], x["beta"], x["h0"], dout, dhT,
                                   *outs, dh0, None, N, T, H, d, d, 16, 2.0, gdr.GDR_BF16,
                                   gdr.GDR_GATE_BOUNDED, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_chunk_bwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, 3)
    breakdown, dom_sel = kernel_breakdown(gdr, torch, step)
    gdr.gdr_profile_select(dom_sel)
    gdr.gdr_profile_read()
    gdr.gdr_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        n0 = gdr.gdr_launch_count()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        n_launch = gdr.gdr_launch_count() - n0
    gdr.gdr_profile_enable(False)
    gdr.gdr_profile_select(None)
    prof = gdr.gdr_profile_read()
    st = gdr.gdr_get_status(stream)
    if st != gdr.GDR_OK:
        raise gdr.GdrError(st, "device status after backward")
    ms = ev0.elapsed_time(ev1) / steps
    dom_name, (dom_ms, dom_n) = max(prof.items(), key=lambda kv: kv[1][0]) if prof else ("?", (0.0, 1))
    flops = 20.0 * d * d * N * T * H
    summ = clk.summary() or {}
    _, bf16_tf, _, peak_src = peaks()
    peak = bf16_tf / 2.0
    achieved = flops / (ms / 1e3) / 1e12
    # bytes: per (token, head) the inputs q, k, v, dout and a, beta, the gradients dq, dk, dv,
    # da, dbeta (a and da carry dk entries with the per-channel gate); per (sequence, head)
    # h0, dhT and dh0.  The chunked form also writes and reads back, per (16-token tile,
    # head), the entering state and the scaled end gradient (bf16) and the tile's delta
    # and its gradient (fp32): scratch, not algorithmic, reported beside it.
    hbm, _, _, _ = peaks()
    ga = 2 * d if vec else 2
    alg_bytes = (2 * (3 * d + d) + ga + 2 + 2 * 3 * d + ga + 2) * N * T * H + 3 * 4 * d * d * N * H
    tiles = N * ((T + 15) // 16)
    scratch_bytes = 2 * tiles * H * (2 * 2 * d * d + 2 * 4 * 16 * d)
    bytes_roof = {"bound": "hbm", "algorithmic_bytes": alg_bytes, "scratch_bytes": scratch_bytes,
                  "achieved": alg_bytes / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                  "frac": alg_bytes / (ms / 1e3) / 1e9 / hbm,
                  "frac_with_scratch": (alg_bytes + scratch_bytes) / (ms / 1e3) / 1e9 / hbm,
                  "t_hbm_ms_with_scratch": (alg_bytes + scratch_bytes) / (hbm * 1e9) * 1e3}
    cpu = None if args.no_cpu else _cpu_line(*cpu_rate_bwd(x, dout, dhT, 2.0, vec, args.cpu_budget),
                                             "sequence 0, its first tokens x 16 heads, with dout and dhT")
    print(json.dumps({
        "metric": ("backward tokens/s, gated delta rule" + (" with per-channel decay" if vec else "")
                   + ", 16 heads, d=128, bf16 in/out, fp32 math"),
        "value": N * T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"backward: N={N} sequences x T={T} x H={H}, dk=dv={d}",
                   "l2_policy": "no flush; the per-step inputs and scratch exceed L2"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "whole step",
                     "peak_source": f"{peak_src} bf16_tflops x 0.5 (tf32)",
                     "algorithmic_flops_per_step": flops, "dominant_kernel": dom_name,
                     "dominant_share": (breakdown[dom_name][0] / sum(v[0] for v in breakdown.values())
                                        if dom_name in breakdown else None)},
        "roofline_bytes": bytes_roof,
        "kernels": kernels_json(breakdown, 2), "kernels_note": KERNELS_NOTE,
        "cpu_baseline": cpu, "gpu_launches": n_launch, "clocks": summ or None,
    }), flush=True)


def bench_vec(args, w):
    """The per-channel decay forward (gdr_chunk_fwd_vec) on the workload's shapes,
    a drawn per key channel.  Algorithmic bytes per (token, head): q, k, v, out and
    the dk gate inputs in the storage dtype plus beta, and the state in and out."""
    import torch
    import chunked_gated_delta_07_gb300 as gdr
    from gdr_inputs import make_channel_gate, make_inputs
    x = make_inputs(w, device="cuda")
    av = make_channel_gate(x, w.seed + 7)
    out = torch.empty_like(x["v"])
    hT = torch.empty((x["N"], w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    dcode = gdr.GDR_BF16 if w.dtype == "bf16" else gdr.GDR_F32
    stream = torch.cuda.current_stream()
    n_tok = x["q"].shape[0] * x["q"].shape[1]

    def step():
        rc = gdr.gdr_chunk_fwd_vec(x["q"], x["k"], x["v"], av, x["beta"], x["h0"], out, hT,
                                   x["cu_seqlens"], x["N"], x["T"], w.H, w.dk, w.dv, 16, w.b,
                                   dcode, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_chunk_fwd_vec")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, 3)
    breakdown, dom_sel = kernel_breakdown(gdr, torch, step)
    gdr.gdr_profile_select(dom_sel)
    gdr.gdr_profile_read()
    gdr.gdr_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        n0 = gdr.gdr_launch_count()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        n_launch = gdr.gdr_launch_count() - n0
    gdr.gdr_profile_enable(False)
    gdr.gdr_profile_select(None)
    prof = gdr.gdr_profile_read()
    st = gdr.gdr_get_status(stream)
    if st != gdr.GDR_OK:
        raise gdr.GdrError(st, "device status after the per-channel forward")
    ms = ev0.elapsed_time(ev1) / steps
    es = 2 if w.dtype == "bf16" else 4
    nstate = x["N"] * w.H * w.dk * w.dv * 4
    byt = n_tok * w.H * (es * (3 * w.dk + 2 * w.dv) + es) + nstate * (2 if x["h0"] is not None else 1)
    hbm, _, _, peak_src = peaks()
    dom_name, (dom_ms, dom_n) = max(prof.items(), key=lambda kv: kv[1][0]) if prof else ("?", (0.0, 1))
    achieved = byt / (ms / 1e3) / 1e9
    cpu = None if args.no_cpu else _cpu_line(*cpu_rate_vec(x, av, w.b, args.cpu_budget),
                                             "the first packed tokens x 16 heads, as one sequence")
    print(json.dumps({
        "metric": "per-channel decay forward tokens/s, bounded gate, bf16 in/out, fp32 state",
        "value": n_tok / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name} with a per key channel: {x['N']} sequences, "
                               f"{n_tok} tokens, H={w.H}, dk=dv={w.dk}, C=16, b={w.b}",
                   "l2_policy": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None, "kernel": "whole step",
                     "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_step": byt,
                     "dominant_kernel": dom_name, "dominant_share":
                         (breakdown[dom_name][0] / sum(v[0] for v in breakdown.values())
                          if dom_name in breakdown else None)},
        "kernels": kernels_json(breakdown, 2), "kernels_note": KERNELS_NOTE,
        "cpu_baseline": cpu, "gpu_launches": n_launch, "clocks": clk.summary(),
    }), flush=True)


def bench_router(args):
    """One statistics window of quantile balancing: zero the counts, route T tokens
    over E = 896 experts (top-k of logit + bias, picked logits returned), then the
    two-sided sign step at q = 0.1 / 0.9.  Algorithmic bytes: the bf16 logits read
    once, the picked indices and logits written, plus the bias and the counts."""
    import torch
    import chunked_gated_delta_07_gb300 as gdr
    from gdr_inputs import make_router_logits
    T, E, k = args.router_tokens, 896, args.router_k
    x, bias = make_router_logits(T, E, 6000, "bf16", device="cuda")
    load = torch.zeros(E, dtype=torch.int64, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    sel = torch.empty((T, k), dtype=torch.float32, device="cuda")
    thr = torch.empty(2, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        load.zero_()
        rc = gdr.gdr_router_topk(x, bias, idx, sel, load, T, E, k, gdr.GDR_BF16, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_router_topk")
        rc = gdr.gdr_router_bias_update(load, bias, thr, E, gdr.GDR_QB_SIGN, 0.1, 0.9, 1e-3, stream)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_router_bias_update")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, 10)
    breakdown, _ = kernel_breakdown(gdr, torch, step)
    gdr.gdr_profile_select("router_topk_kernel")
    gdr.gdr_profile_read()
    gdr.gdr_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        n0 = gdr.gdr_launch_count()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        n_launch = gdr.gdr_launch_count() - n0
    gdr.gdr_profile_enable(False)
    gdr.gdr_profile_select(None)
    prof = gdr.gdr_profile_read()
    ms = ev0.elapsed_time(ev1) / steps
    kern_total, kern_n = prof.get("router_topk_kernel", (0.0, 1))
    kern_ms = kern_total / max(kern_n, 1)
    byt = T * E * 2 + T * k * 8 + E * (4 + 8)
    hbm, _, _, peak_src = peaks()
    achieved = byt / (kern_ms / 1e3) / 1e9 if kern_ms > 0 else 0.0
    cpu = None if args.no_cpu else _cpu_line(*cpu_rate_router(x, bias, k, args.cpu_budget),
                                             "top-k of the window's first tokens")
    print(json.dumps({
        "metric": "router tokens/s, quantile-balancing window (top-8 of 896 experts + bias step)",
        "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"router: T={T} tokens x E={E} experts, k={k}, bf16 logits, "
                               f"sign step q=0.1/0.9",
                   "l2_policy": "logits larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None, "kernel": "router_topk_kernel",
                     "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": byt,
                     "kernel_ms": kern_ms},
        "kernels": kernels_json(breakdown, 2), "kernels_note": KERNELS_NOTE,
        "cpu_baseline": cpu, "gpu_launches": n_launch, "clocks": clk.summary(),
    }), flush=True)


def bench_e2e(gdr, torch, x, w, args, dcode, gcode, pcode, n_tokens):
    """Same metric through gdr_chunk_fwd_host: pinned host inputs in, out and hT back."""
    host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "a", "beta")}
    h0 = x["h0"].cpu().pin_memory() if x["h0"] is not None else None
    cu = x["cu_seqlens"].cpu() if x["cu_seqlens"] is not None else None
    out = torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory()
    hT = torch.empty((x["N"], x["H"], x["dk"], x["dv"]), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    h2d += 0 if h0 is None else h0.numel() * 4
    h2d += 0 if cu is None else cu.numel() * 4
    d2h = out.numel() * out.element_size() + hT.numel() * 4

    def once():
        rc = gdr.gdr_chunk_fwd_host(host["q"], host["k"], host["v"], host["a"], host["beta"], h0,
                                    out, hT, cu, x["N"], x["T"], x["H"], x["dk"], x["dv"], w.chunk,
                                    w.b, dcode, gcode, pcode, None)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_chunk_fwd_host")

    once()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        once()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    return {"value": n_tokens / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": dt * 1e3}


if __name__ == "__main__":
    main()
