"""The N > 1 benchmark path on CPU with gloo, world size 2.

Ranks are independent data-parallel replicas: weights replicated, a batch of
their own, no collective on the data path; only the timing is reduced
(max over ranks) and the throughput counts every rank's tokens. Each rank's
routing must equal a single-process run on that rank's batch (checked with the
oracle), which is what makes the batches independent problems.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as td
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from oracle import Oracle, weights_to_numpy
        from sparse_expert_ffn_softmax_b300 import Workload
        w = Workload("mr_tiny", 40, 16, 32, 4, 2, 1.0, "softmax_topk", "gelu", "f32", has_bias=True)
        t = bench.rank_inputs(w, rank, "cpu")
        # replicated weights, own batch
        wsum = torch.tensor([float(t["w1"].double().sum())], dtype=torch.float64)
        xsum = torch.tensor([float(t["x"].double().sum())], dtype=torch.float64)
        ws = [torch.zeros(1, dtype=torch.float64) for _ in range(WORLD)]
        xs = [torch.zeros(1, dtype=torch.float64) for _ in range(WORLD)]
        td.all_gather(ws, wsum)
        td.all_gather(xs, xsum)
        # per-rank routing on its own batch (no exchange)
        o = Oracle()
        h = weights_to_numpy(t)
        r = o.route(o.config(w), h["x"], o.weights(h))
        # timing: each rank reports its own time; all see the max
        my_ms = 10.0 + 5.0 * rank
        mx = bench.max_over_ranks(my_ms)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), idx=r["idx"], row_of=r["row_of"],
                 wsums=np.array([float(v) for v in ws]), xsums=np.array([float(v) for v in xs]), mx=mx,
                 value=bench.job_tokens_per_s(w.n_tokens, 3, WORLD, mx))
    finally:
        td.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, port, str(tmp_path))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = [np.load(os.path.join(tmp_path, f"rank{r}.npz")) for r in range(WORLD)]
    # weights replicated, batches distinct
    assert res[0]["wsums"][0] == res[0]["wsums"][1]
    assert res[0]["xsums"][0] != res[0]["xsums"][1]
    # max over ranks reaches every rank; throughput counts all ranks' tokens
    assert all(float(r["mx"]) == 15.0 for r in res)
    assert float(res[0]["value"]) == 40 * 3 * 2 / 0.015
    # each rank's routing equals a single-process run on its batch
    import bench
    from oracle import Oracle, weights_to_numpy
    from sparse_expert_ffn_softmax_b300 import Workload
    w = Workload("mr_tiny", 40, 16, 32, 4, 2, 1.0, "softmax_topk", "gelu", "f32", has_bias=True)
    o = Oracle()
    for rank in range(WORLD):
        h = weights_to_numpy(bench.rank_inputs(w, rank, "cpu"))
        r = o.route(o.config(w), h["x"], o.weights(h))
        assert np.array_equal(r["idx"], res[rank]["idx"])
        assert np.array_equal(r["row_of"], res[rank]["row_of"])


# ---- token-sharded batch: the exchange step over gloo, local steps by the oracle ----
SHARD_W = dict(name="shard_tiny", n_tokens=96, d_model=16, d_ff=32, n_experts=6, top_k=2, capacity_factor=0.75,
               gating="softmax_topk", act="gelu", dtype="f32", has_bias=True, logit_bias_max=1.5)
CUTS = (0, 40, 96)  # rank 0: tokens 0-39, rank 1: tokens 40-95
P_SCALE, LSE_SCALE, LSE2_SCALE = 2.0 ** 40, 2.0 ** 32, 2.0 ** 24  # the library's fixed-point statistic words


def _shard_rank(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import sparse_expert_ffn_softmax_b300 as moe
        from oracle import Oracle, weights_to_numpy
        from sparse_expert_ffn_softmax_b300 import Workload
        w = Workload(**SHARD_W)
        h = weights_to_numpy(moe.make_inputs(w, "cpu"))
        a, b = CUTS[rank], CUTS[rank + 1]
        o = Oracle()
        cfg_total = o.config(w)
        C = o.capacity(cfg_total)
        ws_ = w.replace(n_tokens=b - a)
        cfg = o.config(ws_)
        ow = o.weights(h)
        xs = np.ascontiguousarray(h["x"][a:b])
        # step 1 (local): routing and the statistic partial sums of this shard
        L = o.router_logits(cfg, xs, ow)
        idx = o.topk(L, w.top_k)
        gate = o.gates(cfg, L, idx)
        p, lse = o.softmax(L)
        counts = torch.from_numpy(np.bincount(idx.ravel(), minlength=w.n_experts).astype(np.int32))
        words = torch.tensor([int(round(v * P_SCALE)) for v in p.sum(0)] +
                             [int(round(float(lse.sum()) * LSE_SCALE)), int(round(float((lse ** 2).sum()) * LSE2_SCALE))],
                             dtype=torch.int64)
        # step 2: the library's exchange helper over gloo
        shard_counts = moe.exchange_shard_stats(words, counts, None).numpy()
        # step 3 (local): rank base of the earlier shards, then the shard's rows
        base = shard_counts[:rank].sum(0).astype(np.int32)
        r = o.assign_shard(cfg, idx, C, base)
        out = o.outputs(cfg, xs, ow, dict(idx=idx, gate=gate, row_of=r["row_of"]))
        np.savez(os.path.join(out_dir, f"shard{rank}.npz"), idx=idx, gate=gate, row_of=r["row_of"],
                 expert_off=r["expert_off"], kept=r["kept"], dropped=r["dropped"], base=base, out=out,
                 shard_counts=shard_counts, words=words.numpy(), counts=counts.numpy())
    finally:
        td.destroy_process_group()


def test_token_sharded_exchange_equals_unsharded(tmp_path):
    """Two gloo ranks each hold a contiguous token shard of one batch. After the
    exchange (all-gather of per-expert counts, all-reduce of the fixed-point statistic
    sums) and the shard's own capacity step, the top-k, gates, kept (token, choice)
    pairs with their whole-batch ranks, dropped counts, statistics and outputs equal
    the unsharded oracle's."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_shard_rank, args=(r, port, str(tmp_path))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = [np.load(os.path.join(tmp_path, f"shard{r}.npz")) for r in range(WORLD)]
    import sparse_expert_ffn_softmax_b300 as moe
    from oracle import Oracle, weights_to_numpy
    from sparse_expert_ffn_softmax_b300 import Workload
    w = Workload(**SHARD_W)
    h = weights_to_numpy(moe.make_inputs(w, "cpu"))
    o = Oracle()
    cfg = o.config(w)
    ow = o.weights(h)
    full = o.route(cfg, h["x"], ow)
    out_full = o.outputs(cfg, h["x"], ow, full)
    assert full["dropped"] > 0  # the capacity binds, across the shard boundary too
    # every rank got the same exchanged sums; counts are the whole batch's
    for r in res:
        assert np.array_equal(r["counts"], full["counts"])
        assert np.array_equal(r["words"], res[0]["words"])
        assert np.array_equal(r["shard_counts"].sum(0), full["counts"])
    # routing, gates and outputs per token
    assert np.array_equal(np.concatenate([r["idx"] for r in res]), full["idx"])
    assert np.array_equal(np.concatenate([r["gate"] for r in res]), full["gate"])
    assert np.array_equal(np.concatenate([r["out"] for r in res]), out_full)
    # kept pairs and their ranks in the whole batch's token order
    ref, got = {}, {}
    for tt, jj in zip(*np.nonzero(full["row_of"] >= 0)):
        e = int(full["idx"][tt, jj])
        ref[(int(tt), int(jj))] = (e, int(full["row_of"][tt, jj] - full["expert_off"][e]))
    for rank, r in enumerate(res):
        a = CUTS[rank]
        for tt, jj in zip(*np.nonzero(r["row_of"] >= 0)):
            e = int(r["idx"][tt, jj])
            got[(int(a + tt), int(jj))] = (e, int(r["base"][e] + r["row_of"][tt, jj] - r["expert_off"][e]))
    assert got == ref
    assert np.array_equal(sum(r["kept"] for r in res), full["kept"])
    assert sum(int(r["dropped"]) for r in res) == full["dropped"]
    # statistics of the whole batch from the exchanged fixed-point sums
    words = res[0]["words"].astype(np.float64)
    E, N, k = w.n_experts, w.n_tokens, w.top_k
    P = words[:E] / P_SCALE / N
    f = full["counts"] / (N * k)
    st = full["stats"]
    np.testing.assert_allclose(P, st["P"], rtol=1e-9)
    np.testing.assert_allclose(w.aux_alpha * E * np.sum(f * P), st["aux_loss"], rtol=1e-9)
    np.testing.assert_allclose((words[E] / LSE_SCALE / N) ** 2, st["z_loss"], rtol=1e-9)
    np.testing.assert_allclose(words[E + 1] / LSE2_SCALE / N, st["mean_lse_sq"], rtol=1e-6)
