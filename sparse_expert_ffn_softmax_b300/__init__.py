"""Python binding of the sm_103a top-k MoE layer library (``libmoe_b300.so``).

Argument marshalling only: torch supplies device memory and the stream, and
every step of the layer runs in the library's CUDA kernels. The functions have
the C ABI's names (``include/moe.h``) without the ``moe_`` prefix and raise
``MoEError`` on a non-OK status. There is no CPU path: importing this package
raises if the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import torch

from .inputs import ACT, DTYPE, GATING, Workload, WORKLOADS, make_inputs  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_CHECK", 6: "MOE_ERR_TIMEOUT"}


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class moe_config(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("d_model", ctypes.c_int64), ("d_ff", ctypes.c_int64),
                ("n_experts", ctypes.c_int64), ("n_shared", ctypes.c_int64), ("d_ff_shared", ctypes.c_int64),
                ("top_k", ctypes.c_int64), ("capacity_factor", ctypes.c_float), ("gating", ctypes.c_int32),
                ("act", ctypes.c_int32), ("dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("aux_alpha", ctypes.c_float), ("flags", ctypes.c_int32), ("weight_format", ctypes.c_int32),
                ("n_tokens_total", ctypes.c_int64)]


FLAG_DROP_PASSTHROUGH = 1
FLAG_GATHER_ROWS = 2


WEIGHT_FIELDS = ("w_router", "logit_bias", "w1", "w3", "b1", "w2", "b2", "ws1", "ws3", "bs1", "ws2", "bs2",
                 "w1_scale", "w3_scale", "w2_scale")
WEIGHT_FORMAT = {"bf16": 0, "f32": 0, "mxfp8": 1}


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("total_bytes", "status", "logits", "probs", "idx", "gate", "tok_rows", "tok_off", "expert_off",
                 "row_token", "row_gate", "xp", "h", "hs", "yp", "ys", "stats", "stat_acc", "scratch")] + \
               [("max_rows", ctypes.c_int64), ("capacity", ctypes.c_int64)]


class moe_stats_header(ctypes.Structure):
    _fields_ = [("aux_loss", ctypes.c_float), ("z_loss", ctypes.c_float), ("mean_lse_sq", ctypes.c_float),
                ("dropped_share", ctypes.c_float), ("dropped", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("n_experts", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python sparse_expert_ffn_softmax_b300/build.py` "
                          "(the layer has no CPU path)")
    lib = ctypes.CDLL(LIB_PATH)
    P, S = ctypes.c_void_p, ctypes.c_size_t
    c = ctypes.c_int32
    sig = {
        "moe_abi_version": ([], c),
        "moe_status_string": ([c], ctypes.c_char_p),
        "moe_stats_bytes": ([ctypes.c_int64], S),
        "moe_stat_acc_bytes": ([ctypes.c_int64], S),
        "moe_workspace_size": ([P, P], c),
        "moe_workspace_layout_of": ([P, P], c),
        "moe_workspace_init": ([P, P, S, P], c),
        "moe_route": ([P, P, P, P, P, P, P, P, P, S, P], c),
        "moe_permute": ([P, P, P, P, P, P, P, P, P, P, P, P, S, P], c),
        "moe_permute_shard": ([P, P, P, P, P, c, c, P, P, P, P, P, P, P, S, P], c),
        "moe_expert_ffn": ([P, P, P, P, P, P, P, P, P, S, P], c),
        "moe_combine": ([P, P, P, P, P, P, P, P], c),
        "moe_forward": ([P, P, P, P, P, P, S, P], c),
        "moe_forward_traced": ([P, P, P, P, P, P, S, P, P, c], c),
        "moe_forward_overlap": ([P, P, P, P, P, P, S, P, P, P, P, c], c),
        "moe_get_device_status": ([P, P, S, P, P], c),
        "moe_route_noalloc": ([P, P, P, P, P, P, P, P, P], c),
        "moe_get_noalloc_status": ([P, P], c),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def abi_version() -> int:
    return int(_lib.moe_abi_version())


def status_string(code: int) -> str:
    return _lib.moe_status_string(code).decode()


def _check(code: int, where: str):
    if code != 0:
        raise MoEError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---- configuration ----------------------------------------------------------
def config(w: Workload, **over) -> moe_config:
    """moe_config of a workload (see ``inputs.WORKLOADS``); keyword overrides allowed."""
    d = dict(n_tokens=w.n_tokens, d_model=w.d_model, d_ff=w.d_ff, n_experts=w.n_experts, n_shared=w.n_shared,
             d_ff_shared=w.d_ff_shared, top_k=w.top_k, capacity_factor=w.capacity_factor,
             gating=GATING[w.gating], act=ACT[w.act], dtype=DTYPE[w.dtype], has_bias=int(bool(w.has_bias)),
             aux_alpha=w.aux_alpha,
             flags=(FLAG_DROP_PASSTHROUGH if w.drop_passthrough else 0) | (FLAG_GATHER_ROWS if w.gather_rows else 0),
             weight_format=WEIGHT_FORMAT[w.expert_weights], n_tokens_total=0)
    d.update(over)
    return moe_config(**d)


def weights(tensors: Dict[str, Optional[torch.Tensor]]) -> moe_weights:
    """moe_weights from a dict of device tensors (keys as ``inputs.make_inputs``)."""
    mw = moe_weights()
    for n in WEIGHT_FIELDS:
        setattr(mw, n, None if tensors.get(n) is None else _ptr(tensors[n]).value)
    return mw


def stats_bytes(n_experts: int) -> int:
    return int(_lib.moe_stats_bytes(n_experts))


def stat_acc_bytes(n_experts: int) -> int:
    return int(_lib.moe_stat_acc_bytes(n_experts))


def workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(_lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def workspace_layout(cfg: moe_config) -> moe_workspace_layout:
    lay = moe_workspace_layout()
    _check(_lib.moe_workspace_layout_of(ctypes.byref(cfg), ctypes.byref(lay)), "moe_workspace_layout_of")
    return lay


def mx_views(cfg: moe_config, ws: torch.Tensor, region: str):
    """(codes uint8 [max_rows, K], scales uint8 [max_rows, K / 32]) views of the
    workspace's ``xp`` (K = d) or ``h`` (K = F) region of a MOE_WEIGHTS_MXFP8 layer:
    codes first, scales from the next 256-byte boundary (include/moe.h)."""
    lay = workspace_layout(cfg)
    R = int(lay.max_rows)
    K = int(cfg.d_model if region == "xp" else cfg.d_ff)
    base = int(getattr(lay, region))
    off = (R * K + 255) // 256 * 256
    codes = ws[base:base + R * K].view(R, K)
    scales = ws[base + off:base + off + R * (K // 32)].view(R, K // 32)
    return codes, scales


def workspace_init(cfg: moe_config, ws: torch.Tensor, stream=None):
    _check(_lib.moe_workspace_init(ctypes.byref(cfg), _ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def alloc_workspace(cfg: moe_config, device="cuda", stream=None) -> torch.Tensor:
    """A torch-allocated workspace of the required size, with its error word cleared."""
    ws = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=device)
    workspace_init(cfg, ws, stream)
    return ws


def alloc_stats(n_experts: int, device="cuda") -> torch.Tensor:
    return torch.zeros(stats_bytes(n_experts), dtype=torch.uint8, device=device)


def read_stats(buf: torch.Tensor, n_experts: int) -> Dict[str, object]:
    """Decode a device statistics buffer (copies it to the host)."""
    raw = buf.detach().cpu()
    hdr = moe_stats_header.from_buffer_copy(bytes(raw[:ctypes.sizeof(moe_stats_header)].numpy().tobytes()))
    E = n_experts
    body = raw[ctypes.sizeof(moe_stats_header):]
    f = body[:4 * E].view(torch.float32)
    P = body[4 * E:8 * E].view(torch.float32)
    counts = body[8 * E:12 * E].view(torch.int32)
    kept = body[12 * E:16 * E].view(torch.int32)
    out = {n: getattr(hdr, n) for n, _ in moe_stats_header._fields_}
    out.update(f=f.clone(), P=P.clone(), counts=counts.clone(), kept=kept.clone())
    return out


def ws_view(ws: torch.Tensor, offset: int, shape: Sequence[int], dtype: torch.dtype) -> torch.Tensor:
    """A typed view of a workspace region (offsets from ``workspace_layout``)."""
    n = 1
    for s in shape:
        n *= int(s)
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[offset:offset + nbytes].view(dtype).view(*shape)


# ---- stage entry points -----------------------------------------------------
def route(cfg, x, w: moe_weights, idx, gate, logits=None, probs=None, stats=None, ws=None, stream=None):
    _check(_lib.moe_route(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(idx), _ptr(gate), _ptr(logits),
                          _ptr(probs), _ptr(stats), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")


def route_noalloc(cfg, x, w: moe_weights, idx, gate, logits=None, probs=None, stats=None, stream=None):
    """moe_route with no workspace: its scratch is a fixed device array inside the library
    (for callers that cannot allocate; calls must not overlap on the GPU)."""
    _check(_lib.moe_route_noalloc(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(idx), _ptr(gate),
                                  _ptr(logits), _ptr(probs), _ptr(stats), _stream(stream)), "moe_route_noalloc")


def get_noalloc_status(stream=None):
    """(status code, raw error word) of the last route_noalloc call on the current device;
    synchronises the stream and clears the word."""
    word = ctypes.c_int32()
    code = _lib.moe_get_noalloc_status(_stream(stream), ctypes.byref(word))
    return int(code), int(word.value)


def permute(cfg, x, idx, gate, xp, tok_rows, tok_off, expert_off, row_token, row_gate, stats=None, ws=None,
            stream=None):
    _check(_lib.moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(idx), _ptr(gate), _ptr(xp), _ptr(tok_rows),
                            _ptr(tok_off), _ptr(expert_off), _ptr(row_token), _ptr(row_gate), _ptr(stats), _ptr(ws),
                            ws.numel(), _stream(stream)), "moe_permute")


def permute_shard(cfg, x, idx, gate, shard_counts, shard_rank, xp, tok_rows, expert_off, row_token, row_gate,
                  stats=None, ws=None, stream=None):
    _check(_lib.moe_permute_shard(ctypes.byref(cfg), _ptr(x), _ptr(idx), _ptr(gate), _ptr(shard_counts),
                                  int(shard_counts.shape[0]), int(shard_rank), _ptr(xp), _ptr(tok_rows),
                                  _ptr(expert_off), _ptr(row_token), _ptr(row_gate), _ptr(stats), _ptr(ws),
                                  ws.numel(), _stream(stream)), "moe_permute_shard")


def expert_ffn(cfg, xp, expert_off, row_gate, x, w: moe_weights, yp, ys=None, ws=None, stream=None):
    _check(_lib.moe_expert_ffn(ctypes.byref(cfg), _ptr(xp), _ptr(expert_off), _ptr(row_gate), _ptr(x),
                               ctypes.byref(w), _ptr(yp), _ptr(ys), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_ffn")


def combine(cfg, yp, tok_rows, tok_off, ys, out, x=None, stream=None):
    _check(_lib.moe_combine(ctypes.byref(cfg), _ptr(yp), _ptr(tok_rows), _ptr(tok_off), _ptr(ys), _ptr(x), _ptr(out),
                            _stream(stream)), "moe_combine")


def forward(cfg, x, w: moe_weights, out, stats=None, ws=None, stream=None):
    _check(_lib.moe_forward(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(out), _ptr(stats), _ptr(ws),
                            ws.numel(), _stream(stream)), "moe_forward")


def _event_handle(e: torch.cuda.Event, stream) -> ctypes.c_void_p:
    if not e.cuda_event:
        e.record(stream)  # torch creates the CUDA event on its first record
    return ctypes.c_void_p(e.cuda_event)


def forward_overlap(cfg, x, w: moe_weights, out, side_stream, ev_fork: torch.cuda.Event, ev_join: torch.cuda.Event,
                    side_ctas: int = 0, stats=None, ws=None, stream=None):
    """forward with the shared experts' GEMMs on ``side_stream`` (a torch.cuda.Stream),
    forked and joined with the two events; ``side_ctas`` caps their CTAs (0: none)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    _check(_lib.moe_forward_overlap(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(out), _ptr(stats), _ptr(ws),
                                    ws.numel(), _stream(stream), ctypes.c_void_p(side_stream.cuda_stream),
                                    _event_handle(ev_fork, stream), _event_handle(ev_join, stream), int(side_ctas)),
           "moe_forward_overlap")


def forward_traced(cfg, x, w: moe_weights, out, events: Sequence[torch.cuda.Event], stats=None, ws=None,
                   stream=None):
    """forward that records ``events`` (torch.cuda.Event, up to 6) between its stages."""
    if stream is None:
        stream = torch.cuda.current_stream()
    arr = (ctypes.c_void_p * max(1, len(events)))()
    for i, e in enumerate(events):
        if not e.cuda_event:
            e.record(stream)  # torch creates the CUDA event on its first record
        arr[i] = ctypes.c_void_p(e.cuda_event)
    _check(_lib.moe_forward_traced(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(out), _ptr(stats), _ptr(ws),
                                   ws.numel(), _stream(stream), arr, len(events)), "moe_forward_traced")


def get_device_status(cfg, ws, stream=None):
    """(status code, raw error word); synchronises the stream and clears the word."""
    word = ctypes.c_int32()
    code = _lib.moe_get_device_status(ctypes.byref(cfg), _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(word))
    return int(code), int(word.value)


# ---- token-sharded batch (one contiguous token shard per rank) ------------------
def stat_acc_views(cfg, ws: torch.Tensor):
    """The router's statistic partial sums in a workspace: (uint64 words [E + 2] viewed
    as int64 -- fixed-point P sums, lse sum, lse^2 sum --, int32 counts [E])."""
    E = cfg.n_experts
    lay = workspace_layout(cfg)
    acc = ws[lay.stat_acc:lay.stat_acc + stat_acc_bytes(E)]
    return acc[:8 * (E + 2)].view(torch.int64), acc[8 * (E + 2):].view(torch.int32)


def exchange_shard_stats(words: torch.Tensor, counts: torch.Tensor, group=None) -> torch.Tensor:
    """The shards' exchange step: all-gather every shard's per-expert counts (rank
    order) and all-reduce (sum) the fixed-point words and the counts in place.
    Integer sums are exact and independent of the order, so every shard ends with
    the whole batch's sums. Returns shard_counts [world, E] int32."""
    import torch.distributed as td
    world = td.get_world_size(group)
    gathered = [torch.empty_like(counts) for _ in range(world)]
    td.all_gather(gathered, counts.clone(), group=group)
    td.all_reduce(words, op=td.ReduceOp.SUM, group=group)
    td.all_reduce(counts, op=td.ReduceOp.SUM, group=group)
    return torch.stack(gathered)


class ShardBuffers:
    """Views of one shard's intermediates in its workspace (idx, gate, rows, xp, yp, ys)."""

    def __init__(self, cfg, ws: torch.Tensor):
        lay = workspace_layout(cfg)
        N, k, E, d, R = cfg.n_tokens, cfg.top_k, cfg.n_experts, cfg.d_model, lay.max_rows
        dt = torch.bfloat16 if cfg.dtype == DTYPE["bf16"] else torch.float32
        v = lambda off, shape, dtype: ws_view(ws, off, shape, dtype)
        self.idx = v(lay.idx, (N, k), torch.int32)
        self.gate = v(lay.gate, (N, k), torch.float32)
        self.tok_rows = v(lay.tok_rows, (N, k), torch.int32)
        self.expert_off = v(lay.expert_off, (E + 1,), torch.int32)
        self.row_token = v(lay.row_token, (R,), torch.int32)
        self.row_gate = v(lay.row_gate, (R,), torch.float32)
        self.xp = v(lay.xp, (R, d), dt)
        self.yp = v(lay.yp, (R, d), torch.float32)
        self.ys = v(lay.ys, (N, d), torch.float32) if cfg.n_shared > 0 else None


def shard_route(cfg, x, w: moe_weights, ws, stream=None) -> ShardBuffers:
    """Step 1 of a shard: top-k and gates of its tokens; the statistic partial sums stay
    in the workspace for the exchange."""
    b = ShardBuffers(cfg, ws)
    route(cfg, x, w, b.idx, b.gate, None, None, None, ws, stream)
    return b


def shard_finish(cfg, x, w: moe_weights, b: ShardBuffers, shard_counts, shard_rank, out, stats=None, ws=None,
                 stream=None):
    """Steps 3-4 of a shard, after the exchange: rows against the whole batch's capacity,
    statistics of the whole batch, expert FFNs and combine of the shard's tokens."""
    permute_shard(cfg, x, b.idx, b.gate, shard_counts, shard_rank, b.xp, b.tok_rows, b.expert_off, b.row_token,
                  b.row_gate, stats, ws, stream)
    expert_ffn(cfg, b.xp, b.expert_off, b.row_gate, x, w, b.yp, b.ys, ws, stream)
    combine(cfg, b.yp, b.tok_rows, None, b.ys, out, x, stream)


def forward_sharded(cfg, x, w: moe_weights, out, stats=None, ws=None, group=None):
    """This rank's shard of a token-sharded batch (contiguous token ranges in rank order;
    cfg.n_tokens = this shard's tokens, cfg.n_tokens_total = the batch's), on the current
    stream, with the exchange over ``group`` (torch.distributed: NCCL for device tensors).
    Each token's output equals that of the unsharded batch."""
    import torch.distributed as td
    stream = torch.cuda.current_stream()
    b = shard_route(cfg, x, w, ws, stream)
    words, counts = stat_acc_views(cfg, ws)
    shard_counts = exchange_shard_stats(words, counts, group)  # the current stream waits for it
    shard_finish(cfg, x, w, b, shard_counts, td.get_rank(group), out, stats, ws, stream)


class Layer:
    """A layer's config, device weights and workspace, for repeated forwards."""

    def __init__(self, w: Workload, tensors: Dict[str, Optional[torch.Tensor]], device="cuda", **over):
        self.workload = w
        self.cfg = config(w, **over)
        self.tensors = tensors
        self.w = weights(tensors)
        self.layout = workspace_layout(self.cfg)
        self.ws = alloc_workspace(self.cfg, device)
        self.stats = alloc_stats(self.cfg.n_experts, device)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(x)
        forward(self.cfg, x, self.w, out, self.stats, self.ws, stream)
        return out

    def view(self, name: str, shape: Sequence[int], dtype: torch.dtype) -> torch.Tensor:
        return ws_view(self.ws, getattr(self.layout, name), shape, dtype)

    def read_stats(self) -> Dict[str, object]:
        return read_stats(self.stats, self.cfg.n_experts)
