"""moe_route_noalloc -- routing for callers that cannot allocate device memory,
with its scratch in a fixed device array inside the library -- must give the
results of moe_route with a caller workspace, on consecutive calls (the array
keeps the previous call's contents). Collected last on purpose."""
import pytest
import torch

import sparse_expert_ffn_softmax_b300 as moe
from sparse_expert_ffn_softmax_b300 import Workload

CASES = [
    Workload("na_bf16_e8", 1000, 256, 512, 8, 2, 1.25, "softmax_topk_renorm", "gelu", "bf16", has_bias=True),
    Workload("na_bf16_e64_tc", 700, 128, 128, 64, 6, 1.25, "softmax_topk", "swiglu", "bf16", logit_bias_max=2.0),
    Workload("na_f32_ec", 64, 64, 128, 8, 2, 1.0, "expert_choice", "gelu", "f32"),
]


def _route(w, t, noalloc):
    dev = "cuda"
    cfg = moe.config(w)
    E, N = w.n_experts, w.n_tokens
    lay = moe.workspace_layout(cfg)
    C = lay.capacity
    shape = (E, C) if w.gating == "expert_choice" else (N, w.top_k)
    # outputs pre-filled with garbage so a missing write shows up
    idx = torch.full(shape, -7, dtype=torch.int32, device=dev)
    gate = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
    logits = torch.full((N, E), float("nan"), dtype=torch.float32, device=dev)
    probs = torch.full((N, E), float("nan"), dtype=torch.float32, device=dev)
    stats = torch.full((moe.stats_bytes(E),), 0xAB, dtype=torch.uint8, device=dev)
    W = moe.weights(t)
    if noalloc:
        moe.route_noalloc(cfg, t["x"], W, idx, gate, logits, probs, stats)
        assert moe.get_noalloc_status() == (0, 0)  # no device-side condition recorded
    else:
        ws = moe.alloc_workspace(cfg)
        moe.route(cfg, t["x"], W, idx, gate, logits, probs, stats, ws)
    torch.cuda.synchronize()
    return idx, gate, logits, probs, moe.read_stats(stats, E)


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_route(w):
    t = moe.make_inputs(w, "cuda")
    ref = _route(w, t, noalloc=False)
    for _ in range(2):  # the second call starts from the first call's scratch contents
        got = _route(w, t, noalloc=True)
        assert torch.equal(got[0], ref[0])
        torch.testing.assert_close(got[1], ref[1], rtol=1e-5, atol=0)
        torch.testing.assert_close(got[2], ref[2], rtol=1e-5, atol=0)
        torch.testing.assert_close(got[3], ref[3], rtol=1e-5, atol=0)
        for key in ("aux_loss", "z_loss", "mean_lse_sq"):
            assert got[4][key] == pytest.approx(ref[4][key], rel=1e-5)
        torch.testing.assert_close(got[4]["P"], ref[4]["P"], rtol=1e-5, atol=0)
        torch.testing.assert_close(got[4]["f"], ref[4]["f"], rtol=1e-5, atol=0)
        assert torch.equal(got[4]["counts"], ref[4]["counts"])


def test_noalloc_rejects_layers_beyond_its_scratch():
    """The 4 KiB scratch holds the accumulators of at most 318 experts; checked before any launch."""
    w = Workload("na_too_big", 4096, 64, 64, 320, 8, 0.0, "softmax_topk", "gelu", "bf16")
    cfg = moe.config(w)
    fake = torch.empty(0)
    lib = moe._lib
    import ctypes
    p = ctypes.c_void_p(1 << 20)
    W = moe.moe_weights()
    W.w_router = 1 << 20
    code = lib.moe_route_noalloc(ctypes.byref(cfg), p, ctypes.byref(W), p, p, p, None, p, None)
    assert code == 2  # MOE_ERR_UNSUPPORTED
    del fake


@pytest.mark.gpu
def test_noalloc_reports_device_timeout_and_recovers(monkeypatch):
    """A device-side condition during moe_route_noalloc lands in the scratch error word.
    With the single-CTA GEMM's pipeline-wait limit at 1 ns (MOE_GEMM_WAIT_LIMIT_NS), the
    tensor-core logits GEMM of the 64-expert layer (64-wide single-CTA tiles) gives up on its
    first unsatisfied wait and records MOE_ERR_TIMEOUT; moe_get_noalloc_status must report
    it and clear it, and the next call with the normal limit must match moe_route."""
    w = CASES[1]  # na_bf16_e64_tc
    t = moe.make_inputs(w, "cuda")
    ref = _route(w, t, noalloc=False)
    cfg = moe.config(w)
    N, E = w.n_tokens, w.n_experts
    idx = torch.empty((N, w.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((N, w.top_k), dtype=torch.float32, device="cuda")
    logits = torch.empty((N, E), dtype=torch.float32, device="cuda")
    stats = torch.zeros((moe.stats_bytes(E),), dtype=torch.uint8, device="cuda")
    monkeypatch.setenv("MOE_GEMM_WAIT_LIMIT_NS", "1")
    moe.route_noalloc(cfg, t["x"], moe.weights(t), idx, gate, logits, None, stats)
    code, word = moe.get_noalloc_status()
    assert code == 6 and (word & 2), (code, word)  # MOE_ERR_TIMEOUT
    assert moe.get_noalloc_status() == (0, 0)  # read once, cleared
    monkeypatch.delenv("MOE_GEMM_WAIT_LIMIT_NS")
    got = _route(w, t, noalloc=True)  # asserts a clean status itself
    assert torch.equal(got[0], ref[0])
    torch.testing.assert_close(got[1], ref[1], rtol=1e-5, atol=0)
    torch.testing.assert_close(got[2], ref[2], rtol=1e-5, atol=0)
