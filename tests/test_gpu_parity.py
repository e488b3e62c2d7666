"""Parity of the sm_103a library (through its C ABI) with the CPU oracle.

Small layers are compared in full; they span several 128-row GEMM tiles, a
ragged last tile, every gate rule, drops, shared experts, GELU and SwiGLU, fp32
and bf16, the tile widths 64/128/256, and both routers (SIMT dot products;
tensor-core logits, whole or split along K, with the routing kernel). The
workload shapes themselves run at full size with routing compared on every
token; the 8192-token layer and the decode batches compare every output token,
the larger layers 64 sampled tokens plus the expert rows at every expert
segment's ends and in the grouped GEMMs' ragged tiles.
"""
import numpy as np
import pytest
import torch

import sparse_expert_ffn_softmax_b300 as moe
from sparse_expert_ffn_softmax_b300 import WORKLOADS, Workload
from gpu_check import check, run_gpu

pytestmark = pytest.mark.gpu


def wl(name, **kw):
    base = dict(name=name, n_tokens=64, d_model=64, d_ff=128, n_experts=8, top_k=2, capacity_factor=1.25,
                gating="softmax_topk", act="gelu", dtype="bf16", has_bias=False)
    base.update(kw)
    return Workload(**base)


SMALL = [
    WORKLOADS["tiny_f32"],
    wl("f32_swiglu_shared_ec", dtype="f32", act="swiglu", n_shared=2, d_ff_shared=64, gating="expert_choice",
       capacity_factor=1.0, n_tokens=50),
    wl("f32_renorm_drops", dtype="f32", gating="softmax_topk_renorm", capacity_factor=0.5, n_tokens=70,
       has_bias=True),
    wl("bf16_gelu_bias_B", n_tokens=300, d_model=128, d_ff=256, n_experts=4, top_k=2, capacity_factor=1.0,
       gating="topk_softmax", has_bias=True),
    wl("bf16_swiglu_shared", n_tokens=333, d_model=192, d_ff=192, n_experts=6, top_k=3, capacity_factor=1.25,
       act="swiglu", n_shared=2, d_ff_shared=128, logit_bias_max=2.0),
    wl("bf16_gelu_shared_bias", n_tokens=257, d_model=256, d_ff=512, n_experts=5, top_k=2, capacity_factor=0.0,
       gating="softmax_topk_renorm", has_bias=True, n_shared=1, d_ff_shared=256),
    wl("bf16_ec_swiglu", n_tokens=256, d_model=128, d_ff=128, n_experts=8, top_k=2, capacity_factor=1.0,
       gating="expert_choice", act="swiglu", n_shared=1, d_ff_shared=128),
    wl("bf16_k_eq_E", n_tokens=130, d_model=64, d_ff=64, n_experts=3, top_k=3, capacity_factor=0.0),
    wl("bf16_one_expert", n_tokens=129, d_model=128, d_ff=128, n_experts=1, top_k=1, capacity_factor=0.0,
       act="swiglu"),
    wl("bf16_one_token", n_tokens=1, d_model=128, d_ff=256, n_experts=8, top_k=2, capacity_factor=1.25),
    wl("bf16_ragged_tile", n_tokens=33, d_model=64, d_ff=192, n_experts=40, top_k=4, capacity_factor=1.0),
    wl("bf16_many_experts", n_tokens=520, d_model=128, d_ff=128, n_experts=160, top_k=6, capacity_factor=1.25,
       act="swiglu", n_shared=2, d_ff_shared=128, logit_bias_max=2.0),
    wl("bf16_heavy_drops", n_tokens=1000, d_model=64, d_ff=128, n_experts=8, top_k=2, capacity_factor=0.3,
       logit_bias_max=4.0),
    # dropped-token pass-through: tokens with no kept choice (or, in expert choice, picked
    # by no expert) add their input x
    wl("bf16_drops_passthrough", n_tokens=1000, d_model=64, d_ff=128, n_experts=8, top_k=2, capacity_factor=0.3,
       logit_bias_max=4.0, drop_passthrough=True),
    wl("f32_passthrough_shared", dtype="f32", n_tokens=70, capacity_factor=0.4, n_shared=1, d_ff_shared=64,
       has_bias=True, logit_bias_max=3.0, drop_passthrough=True),
    wl("bf16_ec_passthrough", n_tokens=256, d_model=128, d_ff=128, n_experts=8, top_k=2, capacity_factor=0.5,
       gating="expert_choice", act="swiglu", drop_passthrough=True),
    # 16+ token tiles (the router's tile counts and the permute's fused offsets over
    # many blocks): top-2, top-5 of 32 experts with a logit offset, expert choice
    wl("bf16_2k_tokens_B", n_tokens=2100, d_model=128, d_ff=64, n_experts=8, top_k=2, capacity_factor=1.25,
       gating="topk_softmax", has_bias=True),
    wl("bf16_2k_tokens_k5", n_tokens=2049, d_model=64, d_ff=64, n_experts=32, top_k=5, capacity_factor=1.0,
       gating="softmax_topk_renorm", act="swiglu", logit_bias_max=1.0),
    wl("bf16_2k_tokens_ec", n_tokens=2048, d_model=64, d_ff=64, n_experts=12, top_k=2, capacity_factor=1.0,
       gating="expert_choice", act="swiglu", n_shared=1, d_ff_shared=64),
    # tensor-core logits + routing kernel for many experts, with a column count that
    # is not a multiple of 4 and partly filled column chunks
    wl("bf16_E256_k8", n_tokens=300, d_model=128, d_ff=64, n_experts=256, top_k=8, capacity_factor=1.25,
       logit_bias_max=1.0),
    wl("bf16_E33_B", n_tokens=200, d_model=64, d_ff=64, n_experts=33, top_k=5, capacity_factor=1.0,
       gating="topk_softmax"),
    wl("bf16_E129_ec", n_tokens=190, d_model=128, d_ff=64, n_experts=129, top_k=4, capacity_factor=1.0,
       gating="expert_choice"),
    # few token tiles, long K, many experts: the logits GEMM split along K (3 and 4
    # groups here), partial sums added in order by the routing kernel
    wl("bf16_splitk3_router", n_tokens=100, d_model=768, d_ff=64, n_experts=40, top_k=2, capacity_factor=1.25,
       gating="softmax_topk_renorm", act="swiglu"),
    wl("bf16_splitk4_router", n_tokens=200, d_model=1024, d_ff=64, n_experts=64, top_k=4, capacity_factor=1.0,
       logit_bias_max=1.0),
    wl("bf16_k10_two_kernel", n_tokens=150, d_model=64, d_ff=64, n_experts=64, top_k=10, capacity_factor=1.25,
       gating="softmax_topk_renorm"),
    wl("bf16_E300_two_kernel", n_tokens=130, d_model=64, d_ff=64, n_experts=300, top_k=2, capacity_factor=0.0),
    # the SIMT router: bf16 with k > 8 of at most 32 experts, fp32 with more than 64 experts
    wl("bf16_E24_k10_simt", n_tokens=140, d_model=128, d_ff=64, n_experts=24, top_k=10, capacity_factor=1.0,
       gating="softmax_topk_renorm"),
    wl("f32_E72_k3", dtype="f32", n_tokens=90, d_model=64, d_ff=64, n_experts=72, top_k=3, capacity_factor=1.25,
       gating="topk_softmax", has_bias=True),
    # 256-wide down-projection tiles with at least four 128-row tiles per expert: the
    # down-projection runs on CTA pairs (256-row tiles, each CTA staging half of B),
    # odd tile counts leaving the second CTA's half past the expert's rows; the shared
    # experts' K-concatenated down-projection on pairs too
    wl("bf16_pair_gelu_shared_bias", n_tokens=1100, d_model=256, d_ff=512, n_experts=4, top_k=2,
       capacity_factor=1.25, has_bias=True, n_shared=1, d_ff_shared=256),
    wl("bf16_pair_swiglu_ec", n_tokens=1030, d_model=256, d_ff=256, n_experts=4, top_k=2, capacity_factor=1.0,
       gating="expert_choice", act="swiglu", n_shared=2, d_ff_shared=128),
    wl("bf16_pair_skewed", n_tokens=1200, d_model=256, d_ff=256, n_experts=2, top_k=1, capacity_factor=0.0,
       gating="softmax_topk_renorm", logit_bias_max=3.0),
    # the up-projection on CTA pairs (256-wide tiles: experts averaging >= 8 row tiles, or
    # expert choice with C a multiple of 256): SwiGLU with W1 staged by the leader and W3
    # by the peer, ragged last pair tiles, shared experts; GELU + bias in expert choice
    wl("bf16_pair_up_swiglu_shared", n_tokens=2100, d_model=256, d_ff=256, n_experts=2, top_k=1,
       capacity_factor=0.0, act="swiglu", n_shared=1, d_ff_shared=256, logit_bias_max=1.0),
    wl("bf16_pair_up_gelu_bias_ec", n_tokens=1024, d_model=256, d_ff=256, n_experts=4, top_k=2,
       capacity_factor=1.0, gating="expert_choice", has_bias=True),
    # more tiles than CTAs with a last wave at most half full: its tiles are cut into
    # two halves of the tile's columns on two CTAs (183 tiles: up 256 -> 128-column and
    # down 64 -> 32-column halves; 192 tiles: up 64 -> 32, down 256 -> 128 on single CTAs)
    wl("bf16_tail_split", n_tokens=11392, d_model=64, d_ff=256, n_experts=8, top_k=2, capacity_factor=0.0,
       has_bias=True),
    wl("bf16_tail_split_down256", n_tokens=10000, d_model=256, d_ff=64, n_experts=64, top_k=2,
       capacity_factor=0.0, gating="softmax_topk_renorm"),
    # SwiGLU halves: expert choice gives every expert C = 640 rows (5 row tiles), so the
    # up-projection has 8 x 5 x 4 = 160 tiles on 148 SMs and its last 12 become 24 halves
    # of 64 output columns, each two N = 64 MMAs against a quarter of the W1 and W3 halves
    wl("bf16_tail_split_swiglu_ec", n_tokens=2560, d_model=64, d_ff=512, n_experts=8, top_k=2, capacity_factor=1.0,
       gating="expert_choice", act="swiglu"),
    # the tensor-core router (logits GEMM, then the routing kernel) at 16- and 32-token
    # router tiles: every gate rule, ragged last tiles, k = 1 and k = 8, E = 33 .. 256
    wl("bf16_tc_router_renorm", n_tokens=4100, d_model=256, d_ff=128, n_experts=48, top_k=5,
       capacity_factor=1.25, gating="softmax_topk_renorm", act="swiglu", logit_bias_max=2.0),
    wl("bf16_tc_router_B_k8", n_tokens=4096, d_model=128, d_ff=64, n_experts=256, top_k=8, capacity_factor=1.0,
       gating="topk_softmax"),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_layers(w):
    layer, t, res = run_gpu(w)
    check(w, t, res)


def test_tc_router_32_token_tiles():
    """The tensor-core router with 32-token router tiles (batches of >= 16384 tokens), k = 1,
    E = 33, a ragged last tile: routing, gates and statistics on every token, outputs
    on 512 sampled tokens (k = 1 with the renormalised gate, so every output is one
    expert's: the unnormalised top-1 gate makes this narrow layer's outputs so heavy
    tailed that even the exact outputs with bf16 hidden activations miss the bar)."""
    w = wl("bf16_tc_router_k1_tile32", n_tokens=16400, d_model=128, d_ff=128, n_experts=33, top_k=1,
           capacity_factor=1.25, gating="softmax_topk_renorm")
    layer, t, res = run_gpu(w)
    print(check(w, t, res, n_sample=512))


def test_zero_router_ties():
    """All logits equal: every token takes experts 0..k-1, later tokens dropped."""
    w = wl("bf16_zero_router", n_tokens=100, d_model=64, d_ff=128, n_experts=8, top_k=2, capacity_factor=1.0)
    t = moe.make_inputs(w, "cuda")
    t["w_router"].zero_()
    layer, t, res = run_gpu(w, tensors=t)
    assert np.all(res["idx"] == np.arange(2))
    C = res["capacity"]
    assert np.all(res["tok_rows"][C:] == -1)
    check(w, t, res)


def test_empty_batch_is_noop():
    w = wl("bf16_empty", n_tokens=0)
    cfg = moe.config(w)
    t = moe.make_inputs(w.replace(n_tokens=1), "cuda")
    ws = moe.alloc_workspace(cfg)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    moe.forward(cfg, x, moe.weights(t), out, None, ws)
    torch.cuda.synchronize()


def test_deterministic():
    w = WORKLOADS["small_bf16"].replace(n_tokens=2048)
    t = moe.make_inputs(w, "cuda")
    layer = moe.Layer(w, t)
    a = layer.forward(t["x"]).clone()
    st_a = layer.read_stats()
    b = layer.forward(t["x"]).clone()
    st_b = layer.read_stats()
    assert torch.equal(a, b)
    assert st_a["aux_loss"] == st_b["aux_loss"] and torch.equal(st_a["P"], st_b["P"])


def test_stage_calls_match_forward():
    """route -> permute -> expert_ffn -> combine through the separate entry points equals forward."""
    w = wl("bf16_stages", n_tokens=300, d_model=128, d_ff=256, n_experts=6, top_k=2, capacity_factor=1.0,
           act="swiglu", n_shared=1, d_ff_shared=128)
    t = moe.make_inputs(w, "cuda")
    layer = moe.Layer(w, t)
    ref = layer.forward(t["x"]).clone()
    cfg, ws = layer.cfg, layer.ws
    N, k, E, d = w.n_tokens, w.top_k, w.n_experts, w.d_model
    R = layer.layout.max_rows
    dev = "cuda"
    idx = torch.empty(N, k, dtype=torch.int32, device=dev)
    gate = torch.empty(N, k, dtype=torch.float32, device=dev)
    logits = torch.empty(N, E, dtype=torch.float32, device=dev)
    stats = moe.alloc_stats(E)
    moe.route(cfg, t["x"], layer.w, idx, gate, logits, None, stats, ws)
    xp = torch.empty(R, d, dtype=torch.bfloat16, device=dev)
    tok_rows = torch.empty(N, k, dtype=torch.int32, device=dev)
    expert_off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_token = torch.empty(R, dtype=torch.int32, device=dev)
    row_gate = torch.empty(R, dtype=torch.float32, device=dev)
    moe.permute(cfg, t["x"], idx, gate, xp, tok_rows, None, expert_off, row_token, row_gate, stats, ws)
    torch.cuda.synchronize()
    rows = int(expert_off[-1].item())
    assert torch.equal(xp[:rows], t["x"][row_token[:rows].long()])  # permuted rows are exact copies
    yp = torch.empty(R, d, dtype=torch.float32, device=dev)
    ys = torch.empty(N, d, dtype=torch.float32, device=dev)
    moe.expert_ffn(cfg, xp, expert_off, row_gate, t["x"], layer.w, yp, ys, ws)
    out = torch.empty_like(t["x"])
    moe.combine(cfg, yp, tok_rows, None, ys, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert moe.get_device_status(cfg, ws) == (0, 0)


def test_device_index_check_reports():
    """An out-of-range expert id given to moe_permute is caught by the kernels' bounds checks."""
    w = wl("bf16_bad_idx", n_tokens=64, d_model=64, d_ff=128, n_experts=8, top_k=2, capacity_factor=0.0)
    t = moe.make_inputs(w, "cuda")
    cfg = moe.config(w)
    ws = moe.alloc_workspace(cfg)
    N, k, E, d = 64, 2, 8, 64
    R = N * k
    idx = torch.stack([torch.arange(N) % E, (torch.arange(N) + 1) % E], 1).to(torch.int32).cuda()
    idx[5, 1] = 99
    gate = torch.full((N, k), 0.5, device="cuda")
    xp = torch.empty(R, d, dtype=torch.bfloat16, device="cuda")
    tok_rows = torch.empty(N, k, dtype=torch.int32, device="cuda")
    expert_off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.empty(R, dtype=torch.int32, device="cuda")
    row_gate = torch.empty(R, dtype=torch.float32, device="cuda")
    moe.permute(cfg, t["x"], idx, gate, xp, tok_rows, None, expert_off, row_token, row_gate, None, ws)
    code, word = moe.get_device_status(cfg, ws)
    assert code == 5 and (word & 1)
    assert tok_rows[5, 1].item() == -1
    assert moe.get_device_status(cfg, ws) == (0, 0)  # cleared by the read


# (workload, output tokens compared: None = every token). The large layers also
# compare the expert rows of every segment's ends and of the GEMMs' ragged tiles.
FULL = [("small_bf16", None), ("mixtral_decode", None), ("mixtral_prefill", 64), ("fine_skewed", 64),
        ("large_fine", 64), ("large_fine_ec", 64), ("large_fine_decode", None), ("mixtral_decode_fp8", None),
        ("large_fine_decode_fp8", None)]


@pytest.mark.parametrize("name,n_sample", FULL, ids=[f[0] for f in FULL])
def test_full_size_workloads(name, n_sample):
    w = WORKLOADS[name]
    layer, t, res = run_gpu(w)
    rep = check(w, t, res, n_sample=n_sample, raw_bar=True)
    print(name, rep)
    del layer, t, res
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,caps", [("overlap_small", (0, 64)), ("overlap_mxfp8", (0, 64)), ("fine_skewed", (0, 96))])
def test_forward_overlap_matches_forward(name, caps):
    """Shared experts on a second stream (forked at the start of the forward, joined
    before the combine) give the one-stream forward's output bit for bit."""
    if name == "overlap_small":
        w = wl("overlap_small", n_tokens=1500, d_model=256, d_ff=256, n_experts=16, top_k=4, capacity_factor=1.0,
               act="swiglu", n_shared=2, d_ff_shared=256, logit_bias_max=1.0)
    elif name == "overlap_mxfp8":  # MXFP8 routed experts on the main stream, bf16 shared experts beside them
        w = wl("overlap_mxfp8", n_tokens=700, d_model=512, d_ff=512, n_experts=8, top_k=2, capacity_factor=1.0,
               act="swiglu", n_shared=1, d_ff_shared=512, expert_weights="mxfp8")
    else:
        w = WORKLOADS[name]
    t = moe.make_inputs(w, "cuda")
    layer = moe.Layer(w, t)
    ref = layer.forward(t["x"]).clone()
    side = torch.cuda.Stream()
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    for cap in caps:
        out = torch.empty_like(ref)
        for _ in range(2):
            moe.forward_overlap(layer.cfg, t["x"], layer.w, out, side, ev_fork, ev_join, cap, layer.stats, layer.ws)
        torch.cuda.synchronize()
        assert moe.get_device_status(layer.cfg, layer.ws) == (0, 0)
        assert torch.equal(out, ref), cap
    del layer, t
    torch.cuda.empty_cache()


# MXFP8 routed experts (FP8 E4M3 codes, one E8M0 scale per 32 along K; d, F multiples
# of 512): the oracle computes with the exact dequantised weights and rounds each
# routed expert's input and hidden rows to MXFP8 by the same block rule
FP8W = [
    wl("fp8w_swiglu_shared", n_tokens=600, d_model=512, d_ff=1024, n_experts=8, top_k=2, capacity_factor=1.25,
       act="swiglu", n_shared=1, d_ff_shared=256, expert_weights="mxfp8"),
    wl("fp8w_gelu_bias_ec", n_tokens=300, d_model=512, d_ff=512, n_experts=6, top_k=2, capacity_factor=1.0,
       gating="expert_choice", has_bias=True, expert_weights="mxfp8"),
    wl("fp8w_decode_many", n_tokens=40, d_model=1024, d_ff=512, n_experts=64, top_k=6, capacity_factor=0.0,
       act="swiglu", logit_bias_max=1.0, expert_weights="mxfp8"),
    wl("fp8w_drops_passthrough", n_tokens=900, d_model=512, d_ff=512, n_experts=8, top_k=2, capacity_factor=0.6,
       act="swiglu", logit_bias_max=2.0, expert_weights="mxfp8", drop_passthrough=True),
    wl("fp8w_one_token", n_tokens=1, d_model=512, d_ff=512, n_experts=8, top_k=2, capacity_factor=0.0,
       act="swiglu", n_shared=1, d_ff_shared=512, expert_weights="mxfp8"),
    wl("fp8w_ragged_32row_tiles", n_tokens=70, d_model=1536, d_ff=1024, n_experts=12, top_k=3,
       capacity_factor=0.0, gating="topk_softmax", act="gelu", has_bias=True, n_shared=1, d_ff_shared=512,
       expert_weights="mxfp8"),
]


@pytest.mark.parametrize("w", FP8W, ids=lambda w: w.name)
def test_mxfp8_expert_weights(w):
    layer, t, res = run_gpu(w)
    assert t["w1"].dtype == torch.uint8 and t["w1_scale"] is not None
    check(w, t, res)


GATHER = [
    wl("gather_bf16_gelu_bias", n_tokens=1000, d_model=128, d_ff=256, n_experts=6, top_k=2, capacity_factor=1.0,
       gating="topk_softmax", has_bias=True, logit_bias_max=2.0, gather_rows=True),
    wl("gather_bf16_swiglu_shared_ec", n_tokens=700, d_model=256, d_ff=128, n_experts=8, top_k=2,
       capacity_factor=1.0, gating="expert_choice", act="swiglu", n_shared=1, d_ff_shared=128, gather_rows=True),
    wl("gather_bf16_ragged_many", n_tokens=333, d_model=64, d_ff=192, n_experts=40, top_k=4, capacity_factor=1.25,
       gather_rows=True),
]


@pytest.mark.parametrize("w", GATHER, ids=lambda w: w.name)
def test_gather_rows_matches_copy(w):
    """The up-projection reading its rows from x with tile::gather4 (no xp copy) matches
    the oracle and gives the copying forward's output bit for bit."""
    layer, t, res = run_gpu(w)
    assert res["xp"] is None  # no xp region in the workspace
    check(w, t, res)
    copy = moe.Layer(w.replace(gather_rows=False), t)
    assert torch.equal(copy.forward(t["x"]), res["out"].cuda())


def test_gather_rows_full_size_layer():
    """The 8192-token layer, gathered, against the copying forward: every output bit."""
    w = WORKLOADS["small_bf16"]
    t = moe.make_inputs(w, "cuda")
    a = moe.Layer(w.replace(gather_rows=True), t).forward(t["x"])
    b = moe.Layer(w, t).forward(t["x"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["bf16_graph_shared", "mixtral_decode_fp8", "bf16_graph_ec"])
def test_cuda_graph_replay_matches_eager(name):
    """The forward is stream-ordered with no host synchronisation, so it can be captured
    into a CUDA graph: replays of the captured forward (new inputs copied into the same
    buffer in between) give the eager forward's outputs and statistics bit for bit."""
    if name == "mixtral_decode_fp8":
        w = WORKLOADS[name]
    elif name == "bf16_graph_shared":
        w = wl(name, n_tokens=1100, d_model=256, d_ff=512, n_experts=40, top_k=4, capacity_factor=1.0,
               act="swiglu", n_shared=1, d_ff_shared=256, logit_bias_max=1.0)
    else:
        w = wl(name, n_tokens=600, d_model=128, d_ff=256, n_experts=8, top_k=2, capacity_factor=1.0,
               gating="expert_choice", has_bias=True)
    t = moe.make_inputs(w, "cuda")
    layer = moe.Layer(w, t)
    x2 = moe.make_inputs(w, "cuda", with_weights=False, x_seed=7)["x"]
    refs = []
    for x in (t["x"], x2):
        refs.append((layer.forward(x).clone(), layer.read_stats()))
    xbuf = t["x"].clone()
    out = torch.empty_like(xbuf)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture (first launches set kernel attributes)
        moe.forward(layer.cfg, xbuf, layer.w, out, layer.stats, layer.ws, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(layer.cfg, xbuf, layer.w, out, layer.stats, layer.ws, torch.cuda.current_stream())
    for x, (ref_out, ref_st) in zip((t["x"], x2, t["x"]), refs + refs[:1]):
        xbuf.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        st = layer.read_stats()
        for key in ("aux_loss", "z_loss", "dropped", "rows"):
            assert st[key] == ref_st[key], key
        assert torch.equal(st["P"], ref_st["P"]) and torch.equal(st["counts"], ref_st["counts"])
    assert moe.get_device_status(layer.cfg, layer.ws) == (0, 0)
