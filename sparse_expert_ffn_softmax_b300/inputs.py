"""Seeded synthetic workloads for the top-k MoE layer forward.

This module only draws random numbers and names workload shapes; it holds none
of the layer's arithmetic. Both the CUDA path (through the tests and the
benchmark) and the CPU oracle receive the tensors it makes, so it is the one
piece of code they share.

Every tensor is drawn from its own ``torch.Generator`` whose seed is derived
from the workload seed and the tensor's name, so any one tensor can be
re-created alone and the draw does not depend on the order in which tensors
are made. Values are drawn in fp32 and, for bf16 workloads, rounded to bf16
(round-to-nearest-even, as ``Tensor.to`` does). ``N(0, v)`` means variance
``v``: weights are ``N(0, 1/fan_in)``, biases ``N(0, 0.01)`` (std 0.1), the
router weight ``N(0, 1/d)`` and tokens ``N(0, 1)``.

Large weight stacks are drawn one expert at a time so the fp32 staging buffer
stays small; the result does not depend on the device only in the sense that a
given device always gives the same bits for the same seed (CPU and CUDA
generators differ, so parity tests copy the device tensors to the host).
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, Optional

import torch

GATING = {"softmax_topk": 0, "softmax_topk_renorm": 1, "topk_softmax": 2, "expert_choice": 3}
ACT = {"gelu": 0, "swiglu": 1}
DTYPE = {"f32": 0, "bf16": 1}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and routing rule of one MoE layer forward."""

    name: str
    n_tokens: int
    d_model: int
    d_ff: int
    n_experts: int
    top_k: int
    capacity_factor: float  # <= 0: no capacity limit
    gating: str
    act: str
    dtype: str
    has_bias: bool = False
    n_shared: int = 0
    d_ff_shared: int = 0
    logit_bias_max: float = 0.0  # per-expert logit offset rising linearly from 0 to this value
    aux_alpha: float = 0.01
    seed: int = 0
    drop_passthrough: bool = False  # a token with no kept expert row gets x added to its output
    gather_rows: bool = False  # bf16: the up-projection gathers its rows from x (no xp copy)
    expert_weights: str = "bf16"  # routed experts' w1/w3/w2: "bf16" (the layer dtype) or "mxfp8"

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five layer shapes the pages' workloads are modelled on (Mixtral-style
# 8-expert layers and DeepSeek-style fine-grained layers), with the decode and
# expert-choice variants. "tiny_f32" is the small fp32 case that the oracle
# finishes in well under a second.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_f32", 64, 64, 128, 8, 2, 1.25, "softmax_topk", "gelu", "f32", has_bias=True),
        Workload("small_bf16", 8192, 512, 2048, 8, 2, 1.25, "topk_softmax", "gelu", "bf16", has_bias=True),
        Workload("mixtral_prefill", 4096, 4096, 14336, 8, 2, 0.0, "softmax_topk_renorm", "swiglu", "bf16"),
        Workload("mixtral_decode", 64, 4096, 14336, 8, 2, 0.0, "softmax_topk_renorm", "swiglu", "bf16"),
        Workload("fine_skewed", 8192, 5120, 1536, 160, 6, 1.25, "softmax_topk", "swiglu", "bf16",
                 n_shared=2, d_ff_shared=1536, logit_bias_max=2.0),
        Workload("large_fine", 16384, 7168, 2048, 256, 8, 0.0, "softmax_topk", "swiglu", "bf16",
                 n_shared=1, d_ff_shared=2048),
        Workload("large_fine_ec", 16384, 7168, 2048, 256, 8, 1.0, "expert_choice", "swiglu", "bf16",
                 n_shared=1, d_ff_shared=2048),
        Workload("large_fine_decode", 128, 7168, 2048, 256, 8, 0.0, "softmax_topk", "swiglu", "bf16",
                 n_shared=1, d_ff_shared=2048),
        # The decode batches with the routed experts' weights in MXFP8 (FP8 E4M3 codes,
        # one power-of-two scale per 32 along K): half the bytes to stream.
        Workload("mixtral_decode_fp8", 64, 4096, 14336, 8, 2, 0.0, "softmax_topk_renorm", "swiglu", "bf16",
                 expert_weights="mxfp8"),
        Workload("large_fine_decode_fp8", 128, 7168, 2048, 256, 8, 0.0, "softmax_topk", "swiglu", "bf16",
                 n_shared=1, d_ff_shared=2048, expert_weights="mxfp8"),
        # Reduced-expert stand-ins of the two fine-grained layers for profiler captures
        # that must stay a few GB on the device: the same d, F, k, shared experts and
        # rows per expert (16384*8/256 = 512; 8192*6/160 ~ 307), 16 routed experts.
        Workload("large_fine_e16", 1024, 7168, 2048, 16, 8, 0.0, "softmax_topk", "swiglu", "bf16",
                 n_shared=1, d_ff_shared=2048),
        Workload("fine_skewed_e16", 832, 5120, 1536, 16, 6, 1.25, "softmax_topk", "swiglu", "bf16",
                 n_shared=2, d_ff_shared=1536, logit_bias_max=2.0),
        # The large layer's router at full size (16384 tokens, d = 7168, 256 experts,
        # top-8) with small experts (F = 128), so its route stage can be captured alone.
        Workload("large_fine_router", 16384, 7168, 128, 256, 8, 0.0, "softmax_topk", "swiglu", "bf16"),
        Workload("fine_skewed_router", 8192, 5120, 128, 160, 6, 1.25, "softmax_topk", "swiglu", "bf16",
                 logit_bias_max=2.0),
    ]
}

# The layers the benchmark reports, in order (the stand-ins above are for captures only).
BENCH_WORKLOADS = ["tiny_f32", "small_bf16", "mixtral_prefill", "mixtral_decode", "mixtral_decode_fp8", "fine_skewed",
                   "large_fine", "large_fine_ec", "large_fine_decode", "large_fine_decode_fp8"]


def _seed_for(seed: int, name: str) -> int:
    return (seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF


def normal(name: str, shape, std: float, dtype: torch.dtype, device, seed: int = 0,
           chunk_dim0: bool = False) -> torch.Tensor:
    """Seeded N(0, std^2) draw of ``shape``; fp32 draw, then cast to ``dtype``.

    With ``chunk_dim0`` the leading dimension is drawn slice by slice (each slice
    from its own generator), which bounds the fp32 staging memory for stacked
    expert weights.
    """
    device = torch.device(device)
    shape = tuple(int(s) for s in shape)
    if not chunk_dim0 or len(shape) < 2:
        g = torch.Generator(device=device)
        g.manual_seed(_seed_for(seed, name))
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        return t.to(dtype)
    out = torch.empty(shape, dtype=dtype, device=device)
    for i in range(shape[0]):
        g = torch.Generator(device=device)
        g.manual_seed(_seed_for(seed, f"{name}[{i}]"))
        t = torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        out[i].copy_(t)
        del t
    return out


def expert_slice(name: str, i: int, shape, std: float, dtype: torch.dtype, device, seed: int = 0) -> torch.Tensor:
    """Slice ``i`` of a stacked weight drawn with ``chunk_dim0`` (the same bits as
    ``normal(name, (n,) + shape, ..., chunk_dim0=True)[i]``), without drawing the rest."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(_seed_for(seed, f"{name}[{i}]"))
    t = torch.randn(tuple(int(s) for s in shape), generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def mxfp8_quantize(w: torch.Tensor):
    """Block-scaled FP8 copy of a weight matrix [..., K] (K % 32 == 0), the OCP MX
    "MXFP8" format: every 32 consecutive elements along K share one power-of-two scale
    2^(s - 127) (E8M0 byte s) and each element is an FP8 E4M3 code (bias 7, max 448).
    The shared exponent is floor(log2(block max |w|)) - 8, so the block's largest
    element scales into [256, 512) and clamps to 448; elements round to nearest even.
    Returns (codes uint8 [..., K], scales uint8 [..., K / 32]). Input preparation
    only: both the library and the oracle are given these codes."""
    K = w.shape[-1]
    assert K % 32 == 0
    blocks = w.float().reshape(*w.shape[:-1], K // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax)) - 8, torch.zeros_like(amax)).clamp(-100, 100)
    q = (blocks / torch.exp2(e).unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(w.shape)
    scales = (e + 127).to(torch.uint8)
    return codes.contiguous(), scales.contiguous()


def make_inputs(w: Workload, device="cpu", with_weights: bool = True,
                x_seed: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Tokens ``x [N, d]`` and the layer's weights, in nn.Linear ``[out, in]`` layout.

    ``x_seed`` draws the tokens from another seed than the weights (data-parallel
    ranks: replicated weights, a batch of their own).

    Keys: x, w_router [E,d], logit_bias [E] fp32 or None, w1/w3 [E,F,d], b1 [E,F],
    w2 [E,d,F], b2 [E,d], ws1/ws3 [S,Fs,d], bs1 [S,Fs], ws2 [S,d,Fs], bs2 [S,d].
    Absent tensors are None (w3/ws3 for GELU experts, biases when has_bias is off).
    """
    dt = w.torch_dtype
    N, d, F, E, S, Fs = w.n_tokens, w.d_model, w.d_ff, w.n_experts, w.n_shared, w.d_ff_shared
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = normal("x", (N, d), 1.0, dt, device, w.seed if x_seed is None else x_seed)
    if not with_weights:
        return out
    out["w_router"] = normal("w_router", (E, d), 1.0 / math.sqrt(d), dt, device, w.seed)
    if w.logit_bias_max != 0.0:
        out["logit_bias"] = torch.linspace(0.0, w.logit_bias_max, E, dtype=torch.float32, device=device) \
            if E > 1 else torch.zeros(E, dtype=torch.float32, device=device)
    else:
        out["logit_bias"] = None
    big = E * F * d > (1 << 26)
    out["w1"] = normal("w1", (E, F, d), 1.0 / math.sqrt(d), dt, device, w.seed, chunk_dim0=big)
    out["w3"] = normal("w3", (E, F, d), 1.0 / math.sqrt(d), dt, device, w.seed, chunk_dim0=big) \
        if w.act == "swiglu" else None
    out["w2"] = normal("w2", (E, d, F), 1.0 / math.sqrt(F), dt, device, w.seed, chunk_dim0=big)
    if w.expert_weights == "mxfp8":  # the same draws, stored as MXFP8 codes and scales
        for n in ("w1", "w3", "w2"):
            if out[n] is None:
                continue
            src = out[n]
            codes = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
            scales = torch.empty(src.shape[:-1] + (src.shape[-1] // 32,), dtype=torch.uint8, device=src.device)
            for i in range(src.shape[0]):  # one expert at a time: small temporaries
                codes[i], scales[i] = mxfp8_quantize(src[i])
            out[n], out[n + "_scale"] = codes, scales
            del src
    else:
        out["w1_scale"] = out["w3_scale"] = out["w2_scale"] = None
    out["b1"] = normal("b1", (E, F), 0.1, dt, device, w.seed) if w.has_bias else None
    out["b2"] = normal("b2", (E, d), 0.1, dt, device, w.seed) if w.has_bias else None
    if S > 0:
        out["ws1"] = normal("ws1", (S, Fs, d), 1.0 / math.sqrt(d), dt, device, w.seed, chunk_dim0=big)
        out["ws3"] = normal("ws3", (S, Fs, d), 1.0 / math.sqrt(d), dt, device, w.seed, chunk_dim0=big) \
            if w.act == "swiglu" else None
        out["ws2"] = normal("ws2", (S, d, Fs), 1.0 / math.sqrt(Fs), dt, device, w.seed, chunk_dim0=big)
        out["bs1"] = normal("bs1", (S, Fs), 0.1, dt, device, w.seed) if w.has_bias else None
        out["bs2"] = normal("bs2", (S, d), 0.1, dt, device, w.seed) if w.has_bias else None
    else:
        for k in ("ws1", "ws3", "ws2", "bs1", "bs2"):
            out[k] = None
    return out
