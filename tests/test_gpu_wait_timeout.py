"""The grouped GEMM's bounded pipeline waits, made to run out on purpose.

Every mbarrier wait of the GEMM gives up after a time limit (2 s), records
MOE_ERR_TIMEOUT in the workspace error word, lets the CTA's own TMA copies and
MMAs in flight finish (with the full limit), frees its tensor memory and
returns. Here the limit of the single-CTA form is set to 1 ns through
MOE_GEMM_WAIT_LIMIT_NS, so the first wait that is not already satisfied runs
out: the forward must come back, the status must read MOE_ERR_TIMEOUT, and a
following forward with the normal limit on the same workspace must match the
oracle (tensor memory released, no stale state). No wait is left unbounded and
nothing faults: the copies and MMAs the kernel waits for all complete by
themselves.
"""
import pytest

import sparse_expert_ffn_softmax_b300 as moe
from sparse_expert_ffn_softmax_b300 import Workload
from gpu_check import check, run_gpu

pytestmark = pytest.mark.gpu


def test_gemm_wait_timeout_is_reported_and_recovers(monkeypatch):
    # 900 tokens x top-2 over 4 experts: at most 1800 rows, below the 4 x 128 rows per
    # expert at which the down-projection would run on CTA pairs (which keep the 2 s bound)
    w = Workload("bf16_wait_timeout", 900, 256, 512, 4, 2, 1.25, "softmax_topk", "gelu", "bf16", has_bias=True)
    t = moe.make_inputs(w, "cuda")
    layer = moe.Layer(w, t)
    monkeypatch.setenv("MOE_GEMM_WAIT_LIMIT_NS", "1")
    layer.forward(t["x"])
    code, word = moe.get_device_status(layer.cfg, layer.ws)
    assert code == 6 and (word & 2), (code, word)  # MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_GEMM_WAIT_LIMIT_NS")
    layer2, t, res = run_gpu(w, tensors=t, layer=layer)
    check(w, t, res)
    assert moe.get_device_status(layer.cfg, layer.ws) == (0, 0)
