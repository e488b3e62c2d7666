"""bench.py's bookkeeping on the CPU: algorithmic work per forward and the choice of roof."""
import importlib.util
import os

import pytest

from sparse_expert_ffn_softmax_b300 import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PEAKS = dict(hbm=6481.0, bf16=1749.0, bf16_sustained=1366.0, source="measured")


def test_algorithmic_counts(bench):
    w = WORKLOADS["small_bf16"]
    rows = w.n_tokens * w.top_k
    a = bench.algorithmic(w, rows, w.n_experts)
    assert a["up_flops"] == 2 * rows * w.d_model * w.d_ff  # GELU: one projection
    assert a["down_flops"] == a["up_flops"]
    # up reads xp and W1 (+ bias-free byte count) and writes H, each once
    assert a["up_bytes"] == rows * w.d_model * 2 + w.n_experts * w.d_ff * w.d_model * 2 + rows * w.d_ff * 2
    # down reads H and W2 and writes the fp32 gate-scaled rows Yp; the combine reads Yp
    # (fp32) and writes the bf16 output
    assert a["down_bytes"] == rows * w.d_ff * 2 + w.n_experts * w.d_ff * w.d_model * 2 + rows * w.d_model * 4
    assert a["combine_bytes"] == rows * w.d_model * 4 + w.n_tokens * w.d_model * 2 + w.n_tokens * w.top_k * 4
    sw = WORKLOADS["mixtral_prefill"]
    b = bench.algorithmic(sw, sw.n_tokens * sw.top_k, sw.n_experts)
    assert b["up_flops"] == 2 * 2 * sw.n_tokens * sw.top_k * sw.d_model * sw.d_ff  # SwiGLU: W1 and W3
    # shared experts: Ys (fp32) written by the down-projection, read by the combine
    lf = WORKLOADS["large_fine"]
    c = bench.algorithmic(lf, lf.n_tokens * lf.top_k, lf.n_experts)
    N, d, R = lf.n_tokens, lf.d_model, lf.n_tokens * lf.top_k
    assert c["combine_bytes"] == R * d * 4 + N * d * 4 + N * d * 2 + N * lf.top_k * 4
    # MXFP8 experts: weights and routed activations at 1 + 1/32 bytes per element
    fq = WORKLOADS["mixtral_decode_fp8"]
    q = bench.algorithmic(fq, fq.n_tokens * fq.top_k, fq.n_experts)
    bq = 1 + 1 / 32
    R = fq.n_tokens * fq.top_k
    assert q["up_bytes"] == pytest.approx(R * fq.d_model * bq + 8 * 2 * fq.d_ff * fq.d_model * bq + R * fq.d_ff * bq)


@pytest.mark.parametrize("name,bound", [("small_bf16", "tensor"), ("mixtral_prefill", "tensor"),
                                        ("large_fine", "tensor"), ("mixtral_decode", "hbm"),
                                        ("large_fine_decode", "hbm")])
def test_roof_choice(bench, name, bound):
    w = WORKLOADS[name]
    a = bench.algorithmic(w, w.n_tokens * w.top_k, w.n_experts)
    for flops, nbytes in ((a["up_flops"], a["up_bytes"]), (a["down_flops"], a["down_bytes"])):
        r = bench.gemm_roofline(flops, nbytes, 1e-3, PEAKS)
        assert r["bound"] == bound
        assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
        if bound == "hbm":
            assert r["unit"] == "GB/s" and r["achieved"] == pytest.approx(nbytes / 1e-3 / 1e9)
        else:
            assert r["unit"] == "TFLOP/s" and r["achieved"] == pytest.approx(flops / 1e-3 / 1e12)


def test_tensor_peak_choice(bench):
    """Short grouped GEMM launches are measured against the burst bf16 peak, launches of
    more than a millisecond (power-limited clocks) against the sustained one."""
    assert bench.tensor_peak(PEAKS, 0.05)[0] == PEAKS["bf16"]
    assert bench.tensor_peak(PEAKS, 8.0)[0] == PEAKS["bf16_sustained"]
    r = bench.gemm_roofline(1e12, 1e6, 8e-3, PEAKS)
    assert r["peak"] == PEAKS["bf16_sustained"] and r["frac_of_burst"] == pytest.approx(r["achieved"] / PEAKS["bf16"])


def test_sample_sizes_fit_budget(bench):
    w = WORKLOADS["large_fine"]
    n_route, n_ffn = bench.sample_sizes(w, 6.0, (0.02, 1.6, 4, 2))  # 5 ms per routed token, 0.8 s per FFN token
    assert 8 <= n_route <= w.n_tokens and 2 <= n_ffn <= n_route
    assert n_route * 0.005 + n_ffn * 0.8 <= 6.0 * 1.05


def test_reference_arm_runs_without_the_cuda_library():
    """--impl reference times the oracle on the host and never loads libmoe_b300.so."""
    import subprocess
    import sys
    code = ("import sys, json; sys.argv=['bench.py','--impl','reference','--workload','tiny_f32','--steps','2',"
            "'--warmup','1']; import bench; bench.main(); "
            "maps=open('/proc/self/maps').read(); "
            "print(json.dumps({'lib': 'libmoe_b300' in maps, "
            "'pkg': any(m.startswith('sparse_expert_ffn_softmax_b300') for m in sys.modules)}))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    import json
    lines = [json.loads(x) for x in r.stdout.strip().splitlines()]
    ref, probe = lines[0], lines[-1]
    assert ref["impl"] == "reference" and ref["config"]["workload"] == "tiny_f32" and ref["value"] > 0
    assert ref["cpu_baseline"]["cores"] == 1 and ref["cpu_baseline"]["host_cores"] >= 1
    assert probe == {"lib": False, "pkg": False}
