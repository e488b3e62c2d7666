"""The C-ABI library loads on a machine without a GPU, exports what include/moe.h
declares, and rejects bad arguments on the host (no CUDA call is reached)."""
import ctypes
import os
import re

import pytest

import sparse_expert_ffn_softmax_b300 as moe
from sparse_expert_ffn_softmax_b300 import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_symbols_exported():
    names = declared_symbols()
    assert len(names) >= 13, names
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_strings():
    assert moe.abi_version() == 2
    for code in range(7):
        assert moe.status_string(code)
    assert moe.status_string(99) == "unknown status"


def test_struct_sizes_match_header():
    assert ctypes.sizeof(moe.moe_config) == 96
    assert moe.moe_config.n_tokens_total.offset == 88 and moe.moe_config.flags.offset == 80
    assert ctypes.sizeof(moe.moe_weights) == 15 * 8
    assert ctypes.sizeof(moe.moe_stats_header) == 32
    assert moe.stats_bytes(8) == 32 + 16 * 8


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workspace_layout(name):
    w = WORKLOADS[name]
    cfg = moe.config(w)
    lay = moe.workspace_layout(cfg)
    assert lay.total_bytes == moe.workspace_size(cfg)
    offs = [getattr(lay, f) for f, _ in moe.moe_workspace_layout._fields_[1:19]]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and offs[-1] <= lay.total_bytes
    if w.gating == "expert_choice":
        assert lay.capacity == 512 and lay.max_rows == 256 * 512
    else:
        assert lay.max_rows == w.n_tokens * w.top_k
    # the intermediate buffers are large enough for their declared shapes
    b = 4 if w.dtype == "f32" else 2
    assert lay.h - lay.xp >= lay.max_rows * w.d_model * b
    assert lay.hs - lay.h >= lay.max_rows * w.d_ff * b
    if w.dtype == "bf16" and w.expert_weights == "bf16":  # gathering the rows from x: no xp region
        lay_g = moe.workspace_layout(moe.config(w, flags=moe.FLAG_GATHER_ROWS))
        assert lay_g.h - lay_g.xp == 256
        assert lay.total_bytes - lay_g.total_bytes >= lay.max_rows * w.d_model * b - 256


def test_sharded_capacity_follows_the_whole_batch():
    w = WORKLOADS["small_bf16"]
    lay = moe.workspace_layout(moe.config(w, n_tokens=2048, n_tokens_total=8192))
    assert lay.capacity == 2560 and lay.max_rows == 2048 * 2
    assert moe.stat_acc_bytes(8) == 8 * 12 + 16
    assert lay.stat_acc % 256 == 0 and lay.stat_acc + moe.stat_acc_bytes(8) <= lay.scratch


def test_capacity_from_config():
    assert moe.workspace_layout(moe.config(WORKLOADS["tiny_f32"])).capacity == 20
    assert moe.workspace_layout(moe.config(WORKLOADS["small_bf16"])).capacity == 2560
    assert moe.workspace_layout(moe.config(WORKLOADS["fine_skewed"])).capacity == 384
    assert moe.workspace_layout(moe.config(WORKLOADS["mixtral_prefill"])).capacity == 4096


@pytest.mark.parametrize("over,code", [
    (dict(top_k=9), 2),                     # k > E
    (dict(n_experts=600, top_k=2), 2),       # E > 512
    (dict(top_k=0), 1),
    (dict(n_tokens=-1), 1),
    (dict(gating=7), 1),
    (dict(act=1, has_bias=1), 2),           # SwiGLU takes no biases
    (dict(dtype=1, d_model=96), 2),         # bf16 needs d % 64 == 0
    (dict(dtype=1, d_ff=100), 2),
    (dict(capacity_factor=float("nan")), 1),
    (dict(flags=4), 1),                     # unknown flag bit
    (dict(weight_format=5), 1),
    (dict(weight_format=1), 2),             # MXFP8 weights need a bf16 layer with d, F multiples of 512
    (dict(n_tokens_total=10), 1),           # whole batch smaller than the shard
    (dict(gating=3, n_tokens_total=128), 2),  # expert choice is not sharded
])
def test_config_validation(over, code):
    cfg = moe.config(WORKLOADS["tiny_f32"], **over)
    with pytest.raises(moe.MoEError) as e:
        moe.workspace_size(cfg)
    assert e.value.code == code


def test_host_side_argument_errors():
    """Errors found before any launch: bad workspace, null or misaligned pointers."""
    lib = moe._lib
    cfg = moe.config(WORKLOADS["tiny_f32"])
    need = moe.workspace_size(cfg)
    w = moe.moe_weights()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    # workspace too small / null / misaligned
    assert lib.moe_forward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, None, fake, need - 1, None) == 3
    assert lib.moe_forward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, None, None, need, None) == 1
    assert lib.moe_forward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, None, ctypes.c_void_p((1 << 20) + 16),
                           need, None) == 1
    # null router weight
    assert lib.moe_route(ctypes.byref(cfg), fake, ctypes.byref(w), fake, fake, None, None, None, fake, need,
                         None) == 1
    # misaligned tensor pointer
    w.w_router = (1 << 20) + 4
    assert lib.moe_route(ctypes.byref(cfg), fake, ctypes.byref(w), fake, fake, None, None, None, fake, need,
                         None) == 1
    assert lib.moe_workspace_size(None, None) == 1
    # a sharded batch has no one-call forward or unsharded permute; shard ranks are checked
    cfg_s = moe.config(WORKLOADS["tiny_f32"], n_tokens=32, n_tokens_total=64)
    need_s = moe.workspace_size(cfg_s)
    assert lib.moe_forward(ctypes.byref(cfg_s), fake, ctypes.byref(w), fake, None, fake, need_s, None) == 1
    assert lib.moe_permute(ctypes.byref(cfg_s), fake, fake, fake, fake, fake, None, fake, fake, fake, None, fake,
                           need_s, None) == 1
    assert lib.moe_permute_shard(ctypes.byref(cfg_s), fake, fake, fake, fake, 2, 2, fake, fake, fake, fake, fake,
                                 None, fake, need_s, None) == 1
    # pass-through needs the layer input in the combine
    cfg_p = moe.config(WORKLOADS["tiny_f32"], flags=moe.FLAG_DROP_PASSTHROUGH)
    assert lib.moe_combine(ctypes.byref(cfg_p), fake, fake, None, None, None, fake, None) == 1


def test_mxfp8_layer_validation():
    """MXFP8 experts: bf16 layers with d, F multiples of 512, without row gathering;
    xp and h hold codes, then scales from the next 256-byte boundary, inside the
    regions a bf16 layer reserves."""
    w = WORKLOADS["mixtral_decode_fp8"]
    cfg = moe.config(w)
    lay = moe.workspace_layout(cfg)
    R = lay.max_rows
    assert lay.h - lay.xp >= (R * w.d_model + 255) // 256 * 256 + R * w.d_model // 32
    assert lay.hs - lay.h >= (R * w.d_ff + 255) // 256 * 256 + R * w.d_ff // 32
    with pytest.raises(moe.MoEError) as e:
        moe.workspace_size(moe.config(w, flags=moe.FLAG_GATHER_ROWS))
    assert e.value.code == 2
    with pytest.raises(moe.MoEError) as e:
        moe.workspace_size(moe.config(w, d_ff=w.d_ff + 256))
    assert e.value.code == 2
