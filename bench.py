"""Benchmark of the top-k MoE layer forward on B300 (one JSON line on stdout).

A step is one whole forward (route -> permute -> grouped expert FFN -> combine)
of the workload over one batch of seeded synthetic tokens, through the C ABI.
The headline workload is the largest layer that fits one GPU: 16384 tokens,
d = 7168, 256 routed SwiGLU experts (F = 2048, top-8) and one shared expert.
``value`` is whole-job tokens/s with inputs resident in HBM (L2 flushed between
steps by writing a 256 MiB buffer); ``e2e`` is the same forward through the
public API with the tokens copied in from pinned host memory and the output
copied back inside the timed region. Per-stage times come from CUDA events the
library records between its launches on the launching stream. ``per_config``
repeats the measurement (fewer steps, no e2e) on every other workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--no-per-config] [--no-cpu-baseline]

With N > 1 (torchrun), every rank runs its own batch (independent problems,
weak scaling, no collective on the data path); rank 0 prints the max-over-ranks
timing. ``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import importlib.util
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s per config; grouped-GEMM % bf16 peak; permute/combine GB/s"
STAGES = ["route", "permute", "ffn_up", "ffn_down", "combine"]
HEADLINE = "large_fine"
# A grouped GEMM launch longer than this runs long enough for the power limit to
# pull the SM clock down, so it is measured against the sustained bf16 peak.
SUSTAINED_AFTER_MS = 1.0
# CTA caps of the shared experts' side-stream launches timed for moe_forward_overlap (0: none)
OVERLAP_CAPS = (0, 32, 64, 96)


def load_inputs_module():
    """inputs.py by path: the reference arm must not import the package, whose
    __init__ loads the CUDA library."""
    path = os.path.join(ROOT, "sparse_expert_ffn_softmax_b300", "inputs.py")
    spec = importlib.util.spec_from_file_location("moe_bench_inputs", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # (dataclasses look their module up by name)
    spec.loader.exec_module(mod)
    return mod


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

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
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Median SM clock over the samples taken while the GPU was busy (power above
        half of the run's largest draw), the maximum clock and every throttle reason seen."""
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[3])))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": smax, "samples": 0, "reasons": sorted(reasons)}
        pmax = max(p for _, p in rows)
        busy = [c for c, p in rows if p >= 0.5 * pmax] or [c for c, _ in rows]
        return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": smax, "samples": len(rows),
                "samples_under_load": len(busy), "sm_mhz_min_under_load": float(min(busy)),
                "power_w_max": pmax, "reasons": sorted(reasons)}


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the up/down grouped GEMM from the committed ncu capture
    (profiles/gemm_traffic_<workload>.json, scaled to the full launch there when the
    capture ran a reduced stand-in), or None when the GEMM source has changed since."""
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


def config_block(w, world: int) -> dict:
    """The ``config`` object of a line (the same for both arms)."""
    return {"workload": w.name, "n_tokens": w.n_tokens, "d_model": w.d_model, "d_ff": w.d_ff,
            "n_experts": w.n_experts, "n_shared": w.n_shared, "d_ff_shared": w.d_ff_shared, "top_k": w.top_k,
            "capacity_factor": w.capacity_factor, "gating": w.gating, "act": w.act,
            "parallelism": f"dp{world}", "l2": "flushed between steps (256 MiB write)"}


def rank_inputs(w, rank: int, device):
    """A data-parallel rank's inputs: the replicated weights (seed of the workload) and a
    batch of its own (seed of the workload + rank)."""
    import sparse_expert_ffn_softmax_b300 as moe
    return moe.make_inputs(w, device, x_seed=w.seed + rank)


class InputCache:
    """Device inputs per workload; layers of the same shape and seed share their weights
    (the large layer, its expert-choice run and its decode batch; Mixtral prefill and decode)."""

    def __init__(self, moe, dev, rank: int):
        self.moe, self.dev, self.rank = moe, dev, rank
        self.key, self.weights = None, None

    def get(self, w):
        key = (w.d_model, w.d_ff, w.n_experts, w.n_shared, w.d_ff_shared, w.act, w.dtype, w.has_bias,
               w.logit_bias_max, w.seed, w.expert_weights)
        if key != self.key:
            self.key, self.weights = None, None
            torch.cuda.empty_cache()
            t = rank_inputs(w, self.rank, self.dev)
            self.weights = {n: v for n, v in t.items() if n != "x"}
            self.key = key
            return t
        t = dict(self.weights)
        t["x"] = self.moe.make_inputs(w, self.dev, with_weights=False, x_seed=w.seed + self.rank)["x"]
        return t


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
    """Algorithmic FLOPs / bytes per forward (kept rows only, each operand once). The
    gate-scaled expert rows Yp and the shared experts' sum Ys are fp32 for every layer
    dtype; MXFP8 experts read and write their activations as codes plus one scale byte
    per 32."""
    b = 4 if w.dtype == "f32" else 2
    mx = getattr(w, "expert_weights", "bf16") == "mxfp8"
    bw = 1 + 1 / 32 if mx else b  # routed weight bytes per element
    ba = 1 + 1 / 32 if mx else b  # routed experts' activation bytes per element (xp, H)
    m_up = 2 if w.act == "swiglu" else 1
    N, d, F, E, S, Fs, k = w.n_tokens, w.d_model, w.d_ff, w.n_experts, w.n_shared, w.d_ff_shared, w.top_k
    up_flops = 2 * rows * d * F * m_up + 2 * N * d * S * Fs * m_up
    down_flops = 2 * rows * F * d + 2 * N * S * Fs * d
    w_up = touched * F * d * m_up * bw + S * Fs * d * m_up * b
    w_down = touched * d * F * bw + S * d * Fs * b
    return dict(
        up_flops=up_flops, down_flops=down_flops,
        up_bytes=rows * d * ba + N * d * b * (S > 0) + w_up + rows * F * ba + N * S * Fs * b,
        down_bytes=rows * F * ba + N * S * Fs * b + w_down + rows * d * 4 + N * d * 4 * (S > 0),
        route_bytes=N * d * b + E * d * b + N * k * 8 + N * E * 4,
        permute_bytes=N * d * b + rows * d * ba + rows * 8 + N * k * 8,
        combine_bytes=rows * d * 4 + N * d * 4 * (S > 0) + N * d * b + N * k * 4,
    )


def tensor_peak(pk: dict, launch_ms: float):
    """bf16 peak for a grouped GEMM launch of this length: the burst figure for a short
    launch, the sustained (power-limited) one for a launch of more than SUSTAINED_AFTER_MS."""
    if launch_ms > SUSTAINED_AFTER_MS:
        return pk["bf16_sustained"], f"{pk['source']} bf16 dense sustained (launch of {launch_ms:.2f} ms)"
    return pk["bf16"], f"{pk['source']} bf16 dense burst (launch of {launch_ms:.3f} ms)"


def gemm_roofline(flops: float, nbytes: float, seconds: float, pk: dict, traffic=None) -> dict:
    """Roofline entry of a grouped GEMM launch: against whichever roof takes longer at its
    peak -- the bf16 tensor peak for its FLOPs or the HBM bandwidth for its bytes (a decode
    batch streams the expert weights and is bound by the second)."""
    if nbytes / (pk["hbm"] * 1e9) > flops / (pk["bf16"] * 1e12):
        achieved = nbytes / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": traffic, "peak_source": f"{pk['source']} HBM copy"}
    achieved = flops / seconds / 1e12
    peak, src = tensor_peak(pk, seconds * 1e3)
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_of_burst": achieved / pk["bf16"], "traffic": traffic, "peak_source": src}


def launches_per_step(w):
    """Kernels the library launches per forward (the expert-choice memsets not counted)."""
    ec = w.gating == "expert_choice"
    tiles = -(-w.n_tokens // 32)
    # router (+ logits GEMM for bf16 with E > 32); expert choice: statistics finaliser,
    # expert-major probability copy, selection
    route = 1 + (1 if (w.dtype == "bf16" and w.n_experts > 32) else 0) + (3 if ec else 0)
    if ec:
        permute = 4
    else:
        permute = 1 if w.n_experts * tiles <= 8192 else 2
    if w.dtype == "bf16":
        # MXFP8 routed experts run beside separate bf16 launches of the shared experts
        mx = getattr(w, "expert_weights", "bf16") == "mxfp8"
        ffn = 2 * (2 if (mx and w.n_shared > 0) else 1)
    else:
        ffn = 2 * (2 if w.n_shared > 0 else 1)
    return route + permute + ffn + 1


def stage_report(w, stage_avg, rows, touched, pk):
    """Per-stage rates of one workload from its traced stage times (ms)."""
    alg = algorithmic(w, rows, touched)
    s = {k: v / 1e3 for k, v in zip(STAGES, stage_avg)}
    up_tf = alg["up_flops"] / s["ffn_up"] / 1e12
    down_tf = alg["down_flops"] / s["ffn_down"] / 1e12
    rep = {
        "stages_ms": {k: float(v) for k, v in zip(STAGES, stage_avg)},
        "grouped_gemm_tflops": {"up": up_tf, "down": down_tf},
        "grouped_gemm_pct_bf16_peak": {"up": 100 * up_tf / pk["bf16"], "down": 100 * down_tf / pk["bf16"]},
        "grouped_gemm_pct_bf16_sustained": {"up": 100 * up_tf / pk["bf16_sustained"],
                                            "down": 100 * down_tf / pk["bf16_sustained"]},
        "hbm_gbs": {"route": alg["route_bytes"] / s["route"] / 1e9,
                    "permute": alg["permute_bytes"] / s["permute"] / 1e9,
                    "combine": alg["combine_bytes"] / s["combine"] / 1e9,
                    "up": alg["up_bytes"] / s["ffn_up"] / 1e9,
                    "down": alg["down_bytes"] / s["ffn_down"] / 1e9,
                    "peak": pk["hbm"]},
        "rows": int(rows),
        "experts_touched": int(touched),
    }
    rep["hbm_pct"] = {k: 100 * v / pk["hbm"] for k, v in rep["hbm_gbs"].items() if k != "peak"}
    return rep, alg


def measure(moe, w, t, dev, steps, warmup, flush, dist=False):
    """Warm-up, K timed forwards (events around each, L2 flushed before each) and a traced
    pass for per-stage times. Returns (layer, total timed ms, stage averages ms)."""
    layer = moe.Layer(w, t, device=dev)
    x = t["x"]
    out = torch.empty_like(x)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for _ in range(max(3, warmup)):
        moe.forward(layer.cfg, x, layer.w, out, layer.stats, layer.ws)
    torch.cuda.synchronize(dev)
    code, word = moe.get_device_status(layer.cfg, layer.ws)
    if code != 0:
        raise SystemExit(f"{w.name}: device status {code} word {word}")
    if dist:
        import torch.distributed as td
        td.barrier()
    torch.cuda.synchronize(dev)
    # timed steps: one event before and one after each forward (events between the
    # stages would stop each kernel's launch from overlapping the previous one's tail)
    step_ms = []
    for _ in range(steps):
        flush.zero_()
        ev[0].record()
        moe.forward(layer.cfg, x, layer.w, out, layer.stats, layer.ws)
        ev[5].record()
        ev[5].synchronize()
        step_ms.append(ev[0].elapsed_time(ev[5]))
    torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(float(np.sum(step_ms)), dev)
    # per-stage times from a traced pass (events between the stages; their sum exceeds ms_per_step)
    n_traced = max(1, min(steps, 20))
    stage_ms = np.zeros(len(STAGES))
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
        raise SystemExit(f"{w.name}: device status {code} word {word}")
    return layer, out, total_ms, stage_ms / n_traced


def measure_overlap(moe, layer, x, flush, steps, caps):
    """ms per forward with the shared experts on a side stream (moe_forward_overlap), per
    CTA cap of the side launches, against the one-stream forward timed in the same loop
    (the variants take turns, so clock and power changes fall on all of them alike)."""
    out = torch.empty_like(x)
    side = torch.cuda.Stream()
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    variants = [None] + list(caps)

    def run(v):
        if v is None:
            moe.forward(layer.cfg, x, layer.w, out, layer.stats, layer.ws)
        else:
            moe.forward_overlap(layer.cfg, x, layer.w, out, side, ev_fork, ev_join, v, layer.stats, layer.ws)

    for v in variants:
        for _ in range(2):
            run(v)
    torch.cuda.synchronize()
    tot = {v: 0.0 for v in variants}
    for _ in range(steps):
        for v in variants:
            flush.zero_()
            t0.record()
            run(v)
            t1.record()
            t1.synchronize()
            tot[v] += t0.elapsed_time(t1)
    return {"one_stream_ms": tot[None] / steps,
            "side_stream_ms_by_cta_cap": {str(c): tot[c] / steps for c in caps}}


# ---------------------------------------------------------------------------------------
# CPU oracle legs (the oracle as it stands, single-threaded, pinned to one host core)

class PinnedToOneCore:
    """Pins the calling thread to one host core (the sched_setaffinity call that taskset
    makes) for the oracle's timing, and restores the previous mask."""

    def __enter__(self):
        self.prev = os.sched_getaffinity(0)
        self.core = max(self.prev)
        os.sched_setaffinity(0, {self.core})
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.prev)


def oracle_sample_times(w, x_np, host_router, expert_weights_for, n_route, n_ffn, seed):
    """The oracle on a sample of the workload: routing (logits, softmax, top-k, gates,
    capacity) of n_route tokens, and the expert FFN + combine of n_ffn of them.
    expert_weights_for(experts) gives host arrays of the routed experts listed (and the
    shared experts). Returns (route seconds, ffn seconds, tokens routed, tokens through the FFN)."""
    from oracle import Oracle
    o = Oracle()
    rs = np.random.RandomState(seed)
    tok = np.sort(rs.choice(w.n_tokens, n_route, replace=False))
    xs = np.ascontiguousarray(x_np[tok])
    cfg = o.config(w, n_tokens=n_route)
    ow = o.weights(host_router)
    t0 = time.perf_counter()
    r = o.route(cfg, xs, ow)
    t1 = time.perf_counter()
    ffn_tok = np.sort(rs.choice(n_route, n_ffn, replace=False))
    if w.gating == "expert_choice":
        experts = sorted({e for e in range(w.n_experts) if np.isin(r["sel"][e], ffn_tok).any()})
    else:
        experts = sorted(set(r["idx"][ffn_tok].ravel().tolist()))
    h = expert_weights_for(experts)
    remap = np.full(w.n_experts, -1, np.int32)
    remap[experts] = np.arange(len(experts), dtype=np.int32)
    r_out = dict(r)
    if w.gating == "expert_choice":
        r_out["sel"] = np.ascontiguousarray(r["sel"][experts])
        r_out["gate_ec"] = np.ascontiguousarray(r["gate_ec"][experts])
    else:
        r_out["idx"] = np.ascontiguousarray(remap[r["idx"]])
    cfg_out = o.config(w, n_tokens=n_route, n_experts=len(experts))
    ow_out = o.weights(h)
    t2 = time.perf_counter()
    o.outputs(cfg_out, xs, ow_out, r_out, ffn_tok)
    t3 = time.perf_counter()
    return t1 - t0, t3 - t2


def device_expert_weights(w, t):
    """expert_weights_for() over device tensors: host copies of the listed experts only."""
    from oracle import torch_to_numpy

    from oracle import as_bf16_bits, mxfp8_dequant

    def get(experts):
        h = {}
        for n in ("w1", "w3", "b1", "w2", "b2"):
            if t.get(n) is not None:
                sel = torch.as_tensor(experts, device=t[n].device, dtype=torch.long)
                if t.get(n + "_scale") is not None:  # MXFP8: the oracle takes the exact dequantised values
                    h[n] = as_bf16_bits(mxfp8_dequant(t[n][sel].cpu().numpy(), t[n + "_scale"][sel].cpu().numpy()))
                else:
                    h[n] = torch_to_numpy(t[n][sel])
        for n in ("ws1", "ws3", "bs1", "ws2", "bs2"):
            if t.get(n) is not None:
                h[n] = torch_to_numpy(t[n])
        return h
    return get


def sample_sizes(w, budget_s, probe):
    """(tokens to route, tokens through the FFN) so that one sample takes about budget_s,
    from a probe run's per-token times."""
    r_s, f_s, n_r, n_f = probe
    per_r = max(r_s / n_r, 1e-7)
    per_f = max(f_s / n_f, 1e-6)
    n_route = int(min(w.n_tokens, max(8, 0.25 * budget_s / per_r)))
    n_ffn = int(min(n_route, max(2, 0.75 * budget_s / per_f)))
    return n_route, n_ffn


def cpu_oracle_baseline(w, x_np, host_router, weights_for, budget_s=15.0, steps=1, warmup=0, seed=1):
    """Timed oracle samples, pinned to one core. Returns (tokens/s, mean step seconds,
    sample description, core id)."""
    with PinnedToOneCore() as pin:
        n0 = min(w.n_tokens, 16)
        r_s, f_s = oracle_sample_times(w, x_np, host_router, weights_for, n0, 2, seed=0)
        n_route, n_ffn = sample_sizes(w, budget_s, (r_s, f_s, n0, 2))
        for i in range(warmup):
            oracle_sample_times(w, x_np, host_router, weights_for, n_route, n_ffn, seed=100 + i)
        tot_r = tot_f = 0.0
        for i in range(steps):
            r_s, f_s = oracle_sample_times(w, x_np, host_router, weights_for, n_route, n_ffn, seed=seed + i)
            tot_r += r_s
            tot_f += f_s
        per_token = tot_r / steps / n_route + tot_f / steps / n_ffn
        nproc = os.cpu_count() or 1
        sample = (f"per step: routing (logits, softmax, top-k, gates, capacity) of {n_route} of the {w.n_tokens} "
                  f"tokens ({tot_r / steps:.2f} s) + expert FFNs and combine of {n_ffn} of them "
                  f"({tot_f / steps:.2f} s); tokens/s = 1 / (route s per token + FFN s per token); "
                  f"single-threaded fp64 C++ oracle pinned to host core {pin.core} (1 of {nproc} cores)")
        return 1.0 / per_token, (tot_r + tot_f) / steps, sample, nproc


# ---------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = world > 1
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, world)
        return

    import sparse_expert_ffn_softmax_b300 as moe
    from sparse_expert_ffn_softmax_b300 import WORKLOADS
    from sparse_expert_ffn_softmax_b300.inputs import BENCH_WORKLOADS
    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if dist:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=dev)
    pk = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cache = InputCache(moe, dev, rank)

    # ---- the headline workload ----
    t = cache.get(w)
    clk = ClockSampler(local).__enter__()  # from the warm-up to the end of the timed loops
    layer, out, total_ms, stage_avg = measure(moe, w, t, dev, args.steps, args.warmup, flush, dist)
    x = t["x"]
    # ---- end to end through the public API: pinned host tokens in, output back ----
    # Every step copies its tokens in from pinned host memory and its output back;
    # the copies of neighbouring steps overlap the forward on their own streams
    # (step i's H2D and i-1's D2H run while step i-1 / i computes), as a serving loop would.
    e2e_ms = run_e2e(moe, layer, x, args.steps, dev)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    clk.__exit__(None, None, None)

    st = layer.read_stats()
    rows = int(st["rows"])
    touched = int((st["kept"].numpy() > 0).sum())
    rep, alg = stage_report(w, stage_avg, rows, touched, pk)
    overlap = measure_overlap(moe, layer, x, flush, min(args.steps, 10), OVERLAP_CAPS) \
        if w.n_shared > 0 and w.dtype == "bf16" else None
    # dominant kernel: the larger of the two grouped-GEMM launches
    gi = 2 if stage_avg[2] >= stage_avg[3] else 3
    flops = alg["up_flops"] if gi == 2 else alg["down_flops"]
    gbytes = alg["up_bytes"] if gi == 2 else alg["down_bytes"]
    roof = gemm_roofline(flops, gbytes, stage_avg[gi] / 1e3, pk,
                         measured_traffic(w.name, "up" if gi == 2 else "down"))
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
        "config": config_block(w, world),
        "roofline": {"kernel": "grouped_gemm " + ("up" if gi == 2 else "down"), **roof},
        **rep,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(x.numel() * b),
                "d2h_bytes_per_step": int(out.numel() * b)},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clk.summary(),
    }
    if overlap:
        line["shared_on_side_stream_ms"] = overlap
    cpu_inputs = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        from oracle import torch_to_numpy
        cpu_inputs = (torch_to_numpy(t["x"]),
                      {n: (None if t.get(n) is None else torch_to_numpy(t[n])) for n in ("w_router", "logit_bias")},
                      device_expert_weights(w, t))
    del layer, out
    # ---- every other workload, fewer steps, no e2e ----
    if not args.no_per_config:
        per = {w.name: {"tokens_per_s": value, "ms_per_step": total_ms / args.steps, **rep,
                        "clocks": line["clocks"]}}
        # layers that share the headline's weights first (no second draw of them)
        same = lambda v: (v.d_model, v.d_ff, v.n_experts, v.n_shared, v.act, v.expert_weights) == \
            (w.d_model, w.d_ff, w.n_experts, w.n_shared, w.act, w.expert_weights)
        order = sorted((n for n in BENCH_WORKLOADS if n != w.name), key=lambda n: not same(WORKLOADS[n]))
        for name in order:
            wc = WORKLOADS[name]
            tc = cache.get(wc)
            steps_c = min(args.steps, 10)
            clk_c = ClockSampler(local).__enter__()
            lc, _, tot_c, stage_c = measure(moe, wc, tc, dev, steps_c, 3, flush, dist)
            ov = measure_overlap(moe, lc, tc["x"], flush, steps_c, OVERLAP_CAPS) \
                if wc.n_shared > 0 and wc.dtype == "bf16" and wc.n_tokens >= 4096 else None
            clk_c.__exit__(None, None, None)
            stc = lc.read_stats()
            rc, _ = stage_report(wc, stage_c, int(stc["rows"]), int((stc["kept"].numpy() > 0).sum()), pk)
            per[name] = {"tokens_per_s": job_tokens_per_s(wc.n_tokens, steps_c, world, tot_c),
                         "ms_per_step": tot_c / steps_c, "steps": steps_c, **rc,
                         "gpu_launches": launches_per_step(wc) * steps_c, "clocks": clk_c.summary()}
            if ov:
                per[name]["shared_on_side_stream_ms"] = ov
            del lc, tc
        line["per_config"] = per
    if cpu_inputs is not None:
        v, _, sample, nproc = cpu_oracle_baseline(w, *cpu_inputs)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "host_cores": nproc, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        td.destroy_process_group()


def run_reference(args, world):
    """The reference arm: the CPU oracle, as it stands, on one host core, on the same
    workload; each step a bounded sample of it (see cpu_oracle_baseline). The CUDA
    library is not loaded: the inputs come from inputs.py loaded by path, drawn on the
    CPU, and only the experts a sample touches are drawn."""
    inp = load_inputs_module()
    w = inp.WORKLOADS[args.workload]
    from oracle import torch_to_numpy
    import math as _m
    dt = w.torch_dtype
    x = torch_to_numpy(inp.normal("x", (w.n_tokens, w.d_model), 1.0, dt, "cpu", w.seed))
    wr = torch_to_numpy(inp.normal("w_router", (w.n_experts, w.d_model), 1.0 / _m.sqrt(w.d_model), dt, "cpu",
                                   w.seed))
    lb = None
    if w.logit_bias_max != 0.0:
        lb = torch.linspace(0.0, w.logit_bias_max, w.n_experts, dtype=torch.float32).numpy() if w.n_experts > 1 \
            else np.zeros(w.n_experts, np.float32)
    chunked = w.n_experts * w.d_ff * w.d_model > (1 << 26)
    full = None if chunked else inp.make_inputs(w, "cpu")
    shared = {}
    if full is not None:
        shared = {n: torch_to_numpy(full[n]) for n in ("ws1", "ws3", "bs1", "ws2", "bs2") if full.get(n) is not None}
    elif w.n_shared > 0:
        S, Fs, d = w.n_shared, w.d_ff_shared, w.d_model
        specs = [("ws1", (S, Fs, d), 1.0 / _m.sqrt(d)), ("ws2", (S, d, Fs), 1.0 / _m.sqrt(Fs))]
        if w.act == "swiglu":
            specs.append(("ws3", (S, Fs, d), 1.0 / _m.sqrt(d)))
        shared = {n: torch_to_numpy(inp.normal(n, shp, sd, dt, "cpu", w.seed, chunk_dim0=True))
                  for n, shp, sd in specs}
        if w.has_bias:
            shared["bs1"] = torch_to_numpy(inp.normal("bs1", (S, Fs), 0.1, dt, "cpu", w.seed))
            shared["bs2"] = torch_to_numpy(inp.normal("bs2", (S, d), 0.1, dt, "cpu", w.seed))

    def weights_for(experts):
        if full is not None:
            from oracle import as_bf16_bits, mxfp8_dequant
            sel = torch.as_tensor(experts, dtype=torch.long)
            h = {n: (as_bf16_bits(mxfp8_dequant(full[n][sel].numpy(), full[n + "_scale"][sel].numpy()))
                     if full.get(n + "_scale") is not None else torch_to_numpy(full[n][sel]))
                 for n in ("w1", "w3", "b1", "w2", "b2") if full.get(n) is not None}
        else:
            d, F = w.d_model, w.d_ff
            specs = [("w1", (F, d), 1.0 / _m.sqrt(d)), ("w2", (d, F), 1.0 / _m.sqrt(F))]
            if w.act == "swiglu":
                specs.append(("w3", (F, d), 1.0 / _m.sqrt(d)))
            h = {}
            for n, shp, sd in specs:
                v = torch.stack([inp.expert_slice(n, e, shp, sd, dt, "cpu", w.seed) for e in experts])
                if w.expert_weights == "mxfp8":  # the stored codes, as their exact values
                    from oracle import as_bf16_bits, mxfp8_dequant
                    codes, scales = inp.mxfp8_quantize(v)
                    h[n] = as_bf16_bits(mxfp8_dequant(codes.numpy(), scales.numpy()))
                else:
                    h[n] = torch_to_numpy(v)
            if w.has_bias:
                h["b1"] = torch_to_numpy(inp.normal("b1", (w.n_experts, F), 0.1, dt, "cpu", w.seed)[experts])
                h["b2"] = torch_to_numpy(inp.normal("b2", (w.n_experts, d), 0.1, dt, "cpu", w.seed)[experts])
        h.update(shared)
        return h

    # each step is a sample sized so that warm-up + steps take under three minutes
    budget = max(1.0, 140.0 / max(1, args.steps + args.warmup))
    wall0 = time.perf_counter()
    value, step_s, sample, nproc = cpu_oracle_baseline(w, x, {"w_router": wr, "logit_bias": lb}, weights_for,
                                                       budget_s=budget, steps=args.steps, warmup=args.warmup)
    wall = time.perf_counter() - wall0
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)", "config": config_block(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "host_cores": nproc, "kind": "oracle",
                             "sample": sample + "; ms_per_step is the measured time of one sampled step, value "
                                                "the full-batch tokens/s from its per-token times"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
