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
