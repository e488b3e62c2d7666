"""A token-sharded batch on the GPU, shards run one after another in one process.

Each shard routes its contiguous token range (moe_route with n_tokens_total set),
the shards' statistic partial sums and per-expert counts are exchanged (here by
hand: stacked and summed on the device, exactly what the all-gather / all-reduce
of ``exchange_shard_stats`` computes), and each shard then takes its rows against
the whole batch's capacity (moe_permute_shard) and runs its experts and combine.
Nothing waits on another kernel: the shards' launches are simply sequential.
Every token's top-k, gates, kept choices (with their rank in the whole batch),
output and the batch statistics must equal the unsharded forward's bit for bit.
"""
import numpy as np
import pytest
import torch

import sparse_expert_ffn_softmax_b300 as moe
from sparse_expert_ffn_softmax_b300 import Workload
from gpu_check import check, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # drops cross the shard boundary; tensor-core router (E > 32) with a logit offset
    (Workload("shard_bf16_e40", 1024, 128, 128, 40, 4, 1.0, "softmax_topk", "swiglu", "bf16", logit_bias_max=2.0,
              n_shared=1, d_ff_shared=128), (0, 384, 1024)),
    # tensor-core router with 16-token router tiles (shards cut at a router tile's start)
    (Workload("shard_bf16_e64_tile16", 4200, 128, 128, 64, 4, 1.0, "softmax_topk_renorm", "swiglu", "bf16",
              logit_bias_max=2.0), (0, 1008, 4200)),
    # MXFP8 experts: each shard quantises its own rows (xp codes + scales) against the
    # whole batch's capacity
    (Workload("shard_mxfp8_drops", 1536, 512, 512, 8, 2, 0.8, "softmax_topk", "swiglu", "bf16",
              logit_bias_max=2.0, expert_weights="mxfp8"), (0, 512, 1536)),
    # warp-MMA router, GELU with bias, heavy drops, three shards of unequal size
    (Workload("shard_bf16_e8_drops", 2048, 128, 256, 8, 2, 0.5, "topk_softmax", "gelu", "bf16", has_bias=True,
              logit_bias_max=3.0), (0, 640, 672, 2048)),
    # fp32 layer (SIMT router), pass-through of fully dropped tokens
    (Workload("shard_f32_passthrough", 256, 64, 128, 8, 2, 0.4, "softmax_topk_renorm", "gelu", "f32",
              has_bias=True, logit_bias_max=4.0, drop_passthrough=True), (0, 96, 256)),
]


@pytest.mark.parametrize("w,cuts", CASES, ids=[c[0].name for c in CASES])
def test_token_sharded_batch_matches_unsharded(w, cuts):
    N, E, k = w.n_tokens, w.n_experts, w.top_k
    t = moe.make_inputs(w, "cuda")
    layer, t, res = run_gpu(w, tensors=t)
    check(w, t, res)  # the unsharded forward itself against the oracle
    ref_out = res["out"].cuda()
    st_full = res["stats"]
    shards = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        cfg_s = moe.config(w, n_tokens=b - a, n_tokens_total=N)
        ws_s = moe.alloc_workspace(cfg_s)
        x_s = t["x"][a:b].contiguous()
        shards.append((cfg_s, ws_s, x_s, moe.shard_route(cfg_s, x_s, layer.w, ws_s)))
    # the exchange, by hand
    views = [moe.stat_acc_views(c, ws) for c, ws, _, _ in shards]
    shard_counts = torch.stack([cnt.clone() for _, cnt in views])
    words = torch.stack([wd.clone() for wd, _ in views]).sum(0)
    counts = shard_counts.sum(0).to(torch.int32)
    for wd, cnt in views:
        wd.copy_(words)
        cnt.copy_(counts)
    outs, stats = [], []
    for rank, (cfg_s, ws_s, x_s, bufs) in enumerate(shards):
        out_s = torch.empty_like(x_s)
        st = moe.alloc_stats(E)
        moe.shard_finish(cfg_s, x_s, layer.w, bufs, shard_counts, rank, out_s, st, ws_s)
        outs.append(out_s)
        stats.append(moe.read_stats(st, E))
    torch.cuda.synchronize()
    for cfg_s, ws_s, _, _ in shards:
        assert moe.get_device_status(cfg_s, ws_s) == (0, 0)
    assert res["stats"]["dropped"] > 0
    # routing and gates per token
    assert np.array_equal(np.concatenate([b.idx.cpu().numpy() for *_, b in shards]), res["idx"])
    assert np.array_equal(np.concatenate([b.gate.cpu().numpy() for *_, b in shards]), res["gate"])
    # kept choices and their ranks in the whole batch
    off_full = res["expert_off"]
    ref, got = {}, {}
    for tt, jj in zip(*np.nonzero(res["tok_rows"] >= 0)):
        e = int(res["idx"][tt, jj])
        ref[(int(tt), int(jj))] = (e, int(res["tok_rows"][tt, jj] - off_full[e]))
    base = np.zeros(E, np.int64)
    sc = shard_counts.cpu().numpy()
    for rank, (a, (cfg_s, ws_s, x_s, bufs)) in enumerate(zip(cuts, shards)):
        rows = bufs.tok_rows.cpu().numpy()
        idx = bufs.idx.cpu().numpy()
        off = bufs.expert_off.cpu().numpy()
        for tt, jj in zip(*np.nonzero(rows >= 0)):
            e = int(idx[tt, jj])
            got[(int(a + tt), int(jj))] = (e, int(base[e] + rows[tt, jj] - off[e]))
        base += sc[rank]
    assert got == ref
    assert sum(s["dropped"] for s in stats) == st_full["dropped"]
    assert torch.equal(sum(s["kept"] for s in stats), st_full["kept"])
    # the batch statistics, from the exchanged fixed-point sums
    for s in stats:
        for key in ("aux_loss", "z_loss", "mean_lse_sq"):
            assert s[key] == st_full[key], key
        for key in ("f", "P", "counts"):
            assert torch.equal(s[key], st_full[key]), key
    # outputs
    assert torch.equal(torch.cat(outs), ref_out)
