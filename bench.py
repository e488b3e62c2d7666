"""Benchmark of the top-k MoE layer forward on B300 (one JSON line on stdout).

A step is one whole forward (route -> permute -> grouped expert FFN -> combine)
of the workload over one batch of seeded synthetic tokens, through the C ABI.
``value`` is whole-job tokens/s with inputs resident in HBM (L2 flushed between
steps by writing a 256 MiB buffer); ``e2e`` is the same forward through the
public API with the tokens copied in from pinned host memory and the output
copied back inside the timed region. Per-stage times come from CUDA events the
library records between its launches on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 (torchrun), every rank runs its own batch (independent problems,
weak scaling, no collective on the data path); rank 0 prints the max-over-ranks
timing. ``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s per config; grouped-GEMM % bf16 peak; permute/combine GB/s"
STAGES = ["route", "permute", "ffn_up", "ffn_down", "combine"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the up/down grouped GEMM from the committed ncu capture
    (profiles/gemm_traffic_<workload>.json), or None when the GEMM source has changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"gemm_traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    src = os.path.join(ROOT, "sparse_expert_ffn_softmax_b300", "csrc", "gemm_tc.cu")
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != rec.get("gemm_tc_cu_sha256"):
        return None
    return rec.get("traffic_bytes_up" if kernel == "up" else "traffic_bytes_down")


def max_over_ranks(value: float, device=None) -> float:
    """The largest of every rank's value (a single process returns its own)."""
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time (weak scaling)."""
    return tokens_per_rank * steps * world / (max_ms / 1e3)


def rank_inputs(w, rank: int, device):
    """A data-parallel rank's inputs: the replicated weights (seed of the workload) and a
    batch of its own (seed of the workload + rank)."""
    import sparse_expert_ffn_softmax_b300 as moe
    return moe.make_inputs(w, device, x_seed=w.seed + rank)


def run_e2e(moe, layer, x, steps: int, dev) -> float:
    """Milliseconds for `steps` forwards, each with its own pinned H2D of x and D2H of out,
    software-pipelined over three streams with double-buffered device tensors."""
    x_host = x.detach().cpu().pin_memory()
    out_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(x) for _ in range(2)]
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_free[b])  # the forward of step i-2 has read x_dev[b]
            x_dev[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            if i >= 2:
                s_run.wait_event(ev_out[b])  # out_dev[b] of step i-2 has been copied out
            moe.forward(layer.cfg, x_dev[b], layer.w, out_dev[b], layer.stats, layer.ws, stream=s_run)
            ev_free[b].record(s_run)
            ev_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            out_host[b].copy_(out_dev[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(4):  # warm-up
        step(i)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    t1.synchronize()
    return t0.elapsed_time(t1)


def algorithmic(w, rows, touched):
    """Algorithmic FLOPs / bytes per forward (kept rows only, each operand once)."""
    b = 4 if w.dtype == "f32" else 2
    m_up = 2 if w.act == "swiglu" else 1
    N, d, F, E, S, Fs = w.n_tokens, w.d_model, w.d_ff, w.n_experts, w.n_shared, w.d_ff_shared
    up_flops = 2 * rows * d * F * m_up + 2 * N * d * S * Fs * m_up
    down_flops = 2 * rows * F * d + 2 * N * S * Fs * d
    w_up = touched * F * d * m_up * b + S * Fs * d * m_up * b
    w_down = touched * d * F * b + S * d * Fs * b
    return dict(
        up_flops=up_flops, down_flops=down_flops,
        up_bytes=rows * d * b + N * d * b * (S > 0) + w_up + rows * F * b + N * S * Fs * b,
        down_bytes=rows * F * b + N * S * Fs * b + w_down + rows * d * b + N * d * b * (S > 0),
        route_bytes=N * d * b + E * d * b + N * w.top_k * 8 + N * E * 4,
        permute_bytes=N * d * b + rows * d * b + rows * 8 + N * w.top_k * 8,
        combine_bytes=rows * d * b + N * d * b * (2 if S > 0 else 1) + N * w.top_k * 4,
    )


def gemm_roofline(flops: float, nbytes: float, seconds: float, pk: dict, traffic=None) -> dict:
    """Roofline entry of a grouped GEMM launch: against whichever roof takes longer at its
    peak -- the bf16 tensor peak for its FLOPs or the HBM bandwidth for its bytes (a decode
    batch streams the expert weights and is bound by the second)."""
    if nbytes / (pk["hbm"] * 1e9) > flops / (pk["bf16"] * 1e12):
        achieved = nbytes / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": traffic, "peak_source": f"{pk['source']} HBM copy"}
    achieved = flops / seconds / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": achieved / pk["bf16"], "traffic": traffic, "peak_source": f"{pk['source']} bf16 dense burst"}


def launches_per_step(w):
    """Kernels the library launches per forward (the expert-choice bitmap memset not counted)."""
    ec = w.gating == "expert_choice"
    tiles = -(-w.n_tokens // 32)
    route = 1 + (1 if (w.dtype == "bf16" and w.n_experts > 32) else 0) + (2 if ec else 0)
    if ec:
        permute = 4
    else:
        permute = 1 if w.n_experts * tiles <= 8192 else 2
    if w.dtype == "bf16":
        ffn = 2
    else:
        ffn = 2 * (2 if w.n_shared > 0 else 1)
    return route + permute + ffn + 1


def cpu_oracle_step(w, host, n_tokens_sample, seed=0):
    """One oracle pass on a sample: routing of all N tokens + outputs of n sampled tokens.
    Returns (seconds for routing, seconds for the sampled outputs, threads used)."""
    from oracle import Oracle
    o = Oracle()
    cfg = o.config(w)
    ow = o.weights(host)
    t0 = time.perf_counter()
    r = o.route(cfg, host["x"], ow)
    t1 = time.perf_counter()
    rs = np.random.RandomState(seed)
    tokens = np.sort(rs.choice(w.n_tokens, n_tokens_sample, replace=False))
    o.outputs(cfg, host["x"], ow, r, tokens)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def host_copy(t):
    from oracle import weights_to_numpy
    return weights_to_numpy(t)


def run_cpu_baseline(w, host, budget_s=15.0):
    """The oracle as it stands, single-threaded on a host core, on a bounded sample.
    tokens/s = 1 / (route_time / N + ffn_time / n_sample)."""
    r_s, f_s = cpu_oracle_step(w, host, 2)
    per_tok = max(f_s / 2, 1e-6)
    n = int(max(2, min(w.n_tokens, (budget_s - r_s) / per_tok)))
    r_s, f_s = cpu_oracle_step(w, host, n, seed=1)
    value = 1.0 / (r_s / w.n_tokens + f_s / n)
    return dict(value=value, unit="tokens/s", cores=1, kind="oracle",
                sample=f"routing of all {w.n_tokens} tokens ({r_s:.2f} s) + expert FFN and combine of "
                       f"{n} sampled tokens ({f_s:.2f} s); single-threaded fp64 C++")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="small_bf16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    import sparse_expert_ffn_softmax_b300 as moe
    from sparse_expert_ffn_softmax_b300 import WORKLOADS
    w = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = world > 1
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, w)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if dist:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=dev)

    t = rank_inputs(w, rank, dev)
    layer = moe.Layer(w, t, device=dev)
    x = t["x"]
    out = torch.empty_like(x)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]

    clk = ClockSampler(local).__enter__()  # sampled from the warm-up to the end of the timed loops
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        moe.forward(layer.cfg, x, layer.w, out, layer.stats, layer.ws)
    torch.cuda.synchronize(dev)
    code, word = moe.get_device_status(layer.cfg, layer.ws)
    if code != 0:
        raise SystemExit(f"device status {code} word {word}")

    stage_ms = np.zeros(len(STAGES))
    step_ms = []
    if dist:
        td.barrier()
    torch.cuda.synchronize(dev)
    # timed steps: one event before and one after each forward (events between the
    # stages would stop each kernel's launch from overlapping the previous one's tail)
    for _ in range(args.steps):
        flush.zero_()
        ev[0].record()
        moe.forward(layer.cfg, x, layer.w, out, layer.stats, layer.ws)
        ev[5].record()
        ev[5].synchronize()
        step_ms.append(ev[0].elapsed_time(ev[5]))
    torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(float(np.sum(step_ms)), dev)
    # per-stage times from a traced pass (events between the stages; their sum exceeds ms_per_step)
    n_traced = max(1, min(args.steps, 50))
    for _ in range(n_traced):
        flush.zero_()
        moe.forward_traced(layer.cfg, x, layer.w, out, ev, layer.stats, layer.ws)
        ev[-1].synchronize()
        stage_ms += np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(5)])
    torch.cuda.synchronize(dev)
    if dist:
        td.barrier()
    code, word = moe.get_device_status(layer.cfg, layer.ws)
    if code != 0:
        raise SystemExit(f"device status {code} word {word}")

    # ---- end to end through the public API: pinned host tokens in, output back ----
    # Every step copies its tokens in from pinned host memory and its output back;
    # the copies of neighbouring steps overlap the forward on their own streams
    # (step i's H2D and i-1's D2H run while step i-1 / i computes), as a serving loop would.
    e2e_ms = run_e2e(moe, layer, x, args.steps, dev)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    clk.__exit__(None, None, None)

    st = layer.read_stats()
    rows = int(st["rows"])
    kept = st["kept"].numpy()
    touched = int((kept > 0).sum())
    alg = algorithmic(w, rows, touched)
    pk = peaks()
    stage_avg = stage_ms / n_traced
    # dominant kernel: the larger of the two grouped-GEMM launches
    gi = 2 if stage_avg[2] >= stage_avg[3] else 3
    flops = alg["up_flops"] if gi == 2 else alg["down_flops"]
    gbytes = alg["up_bytes"] if gi == 2 else alg["down_bytes"]
    dom_s = stage_avg[gi] / 1e3
    achieved_tflops = flops / dom_s / 1e12
    roof = gemm_roofline(flops, gbytes, dom_s, pk, measured_traffic(w.name, "up" if gi == 2 else "down"))
    value = job_tokens_per_s(w.n_tokens, args.steps, world, total_ms)
    e2e_value = job_tokens_per_s(w.n_tokens, args.steps, world, e2e_ms)
    b = 4 if w.dtype == "f32" else 2
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "n_tokens": w.n_tokens, "d_model": w.d_model, "d_ff": w.d_ff,
                   "n_experts": w.n_experts, "top_k": w.top_k, "capacity_factor": w.capacity_factor,
                   "gating": w.gating, "act": w.act, "n_shared": w.n_shared, "parallelism": f"dp{world}",
                   "l2": "flushed between steps (256 MiB write)"},
        "roofline": {"kernel": "grouped_gemm " + ("up" if gi == 2 else "down"), **roof},
        "stages_ms": {s: float(v) for s, v in zip(STAGES, stage_avg)},
        "grouped_gemm_pct_bf16_peak": {
            "up": 100 * alg["up_flops"] / (stage_avg[2] / 1e3) / 1e12 / pk["bf16"],
            "down": 100 * alg["down_flops"] / (stage_avg[3] / 1e3) / 1e12 / pk["bf16"]},
        "hbm_gbs": {"route": alg["route_bytes"] / (stage_avg[0] / 1e3) / 1e9,
                    "permute": alg["permute_bytes"] / (stage_avg[1] / 1e3) / 1e9,
                    "combine": alg["combine_bytes"] / (stage_avg[4] / 1e3) / 1e9,
                    "up": alg["up_bytes"] / (stage_avg[2] / 1e3) / 1e9,
                    "down": alg["down_bytes"] / (stage_avg[3] / 1e3) / 1e9,
                    "peak": pk["hbm"]},
        "rows": rows,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(x.numel() * b),
                "d2h_bytes_per_step": int(out.numel() * b)},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        host = host_copy(t)
        line["cpu_baseline"] = run_cpu_baseline(w, host)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        td.destroy_process_group()


def run_reference(args, w):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    import sparse_expert_ffn_softmax_b300 as moe
    t = moe.make_inputs(w, "cpu")
    from oracle import weights_to_numpy
    host = weights_to_numpy(t)
    # size each step's sample so the whole run stays within a few minutes
    r_s, f_s = cpu_oracle_step(w, host, 2)
    per_tok = max(f_s / 2, 1e-6)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(2, min(w.n_tokens, (budget - r_s) / per_tok)))
    for i in range(args.warmup):
        cpu_oracle_step(w, host, n, seed=100 + i)
    tot_r = tot_f = 0.0
    for i in range(args.steps):
        r_s, f_s = cpu_oracle_step(w, host, n, seed=i)
        tot_r += r_s
        tot_f += f_s
    per_step_s = tot_r / args.steps + (tot_f / args.steps) * w.n_tokens / n
    value = w.n_tokens / per_step_s
    sample = (f"each step: routing of all {w.n_tokens} tokens + expert FFN/combine of {n} sampled tokens, "
              f"scaled to the full batch; single-threaded fp64 C++ oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "n_tokens": w.n_tokens},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
